/*
 * spec_verify.h -- C ABI of the GB300 speculative-decoding verification sampler.
 *
 * One call verifies a batch of requests: for each request i with K_i draft tokens it takes
 * the target model's logits at the K_i draft positions and at one bonus position, computes
 * p = softmax(logits / T), accepts draft d at position j when u < min(1, p(d) / q(d)), stops at
 * the first rejection and emits there a token drawn from the residual max(0, p - q) (or from p
 * with d removed when no draft distribution is given), or appends a bonus token drawn from p
 * when every draft is accepted. Greedy requests accept iff d is the target argmax.
 *
 * Pages (title, section) the operation is defined by:
 *   [MTP-eagle]    "【vllm】DeepSeekMTP、eagle": sample() call tree -- logits at num_draft + 1
 *                  positions per request, Gumbel-max sampler, _rejection_sample_kernel (one
 *                  program per request, stop at the first mismatch, bonus when all match),
 *                  outputs sampled[num_reqs, num_spec_steps + 1], num_sampled, num_rejected.
 *   [spec-notes]   "vLLM 投机解码（Eagle / MTP）实现与运行流程": residual distribution Q&A
 *                  (min(1, p/q), max(0, p - q) normalised), bonus token and NO_DRAFT_PROBS
 *                  Q&A (accept test code, masked target probs, argmax(prob / Exp(1))),
 *                  section 8.2 (rejection_sample(draft_token_ids, num_draft_tokens,
 *                  draft_probs, target_probs, bonus_token_ids)), 8.3 (greedy / stochastic
 *                  rules), 9.2 (num_rejected = num_draft - num_accepted).
 *   [spec-in-vllm] "speculative decoding in vLLM": 7.0 acceptance u < p/q and residual,
 *                  7.0.1 greedy, 7.0.2 bonus, 7.3 Gumbel argmax, 7.4 stats / reject /
 *                  resample / insert kernels.
 *   [mini-sglang]  "mini-sglang", "how tokens are sampled": temperature <= 0 means greedy.
 *
 * Conventions fixed by this library where the pages leave them open:
 *   - Rows: the logits of (request i, position j), j = 0..K_i (j = K_i is the bonus
 *     position), are row cu_num_draft[i] + i + j of a row-major [num_draft_tokens + num_reqs, V]
 *     array; draft j of request i is draft_ids[cu_num_draft[i] + j] and its distribution is row
 *     cu_num_draft[i] + j of draft_probs [num_draft_tokens, V].
 *   - x_v = logit_v * (1 / T) in binary32; a request is greedy if is_greedy[i] != 0 or
 *     !(T > 0). Greedy argmax is over the raw logits, lowest index on ties.
 *   - Random draws are keyed, so results are reproducible and independent of launch shape:
 *     Philox4x32-10 (Salmon et al., SC'11), key = (lo32(seed), hi32(seed)), counter =
 *     (c0, j, req_index_base + i, tag), uniform U = ((w >> 9) + 1/2) / 2^23 of a 32-bit word w.
 *     The acceptance uniform u of position j is word 0 of counter (0, j, i', 0).
 *   - A draw from weights w_v is the exponential race argmax_v w_v / E_v over i.i.d. Exp(1)
 *     clocks E_v (the key is the binary32 quotient), lowest index on equal keys. The clocks come in groups of 64 tokens
 *     (g = v >> 6, slot s = v & 63): counter (g, j, i', 8) gives W (word 0) and the slot
 *     a = word 1 & 63 that holds the group's smallest clock E_g = -log(W) / 64; slot s != a has
 *     clock E_g + (-log U_s), U_s word s & 3 of counter (g, j, i', 9 + s / 4). (By the
 *     memoryless property these are i.i.d. Exp(1); E_g bounds every key of the group, which
 *     lets the race skip whole groups.) Over p the weights are t_v = exp(x_v - m); residual
 *     weights are rr_v = fma(-S, q_v, t_v) (S times p_v - q_v, rounded once), candidates
 *     rr_v > 0; if no candidate is left after rounding, the token is drawn from p. Without draft
 *     probabilities the rejected draft token is removed.
 *   - Acceptance: 0 <= d < V and q(d) > 0 and p(d) / q(d) >= u (binary32), q(d) = 1 without
 *     draft probabilities. An out-of-range draft id is rejected, not an error.
 *   - exp / log inside these decisions are fixed binary32 functions (Cody-Waite reduction
 *     with a degree-7 Taylor polynomial; atanh series on [sqrt(1/2), sqrt(2))). The one input
 *     they take that is not fixed bit for bit is S, the sum of exponentials: it is summed with
 *     the hardware's approximate 2^x, in an order of the kernel's choosing, and matches the
 *     exactly summed S to about 1e-6 relative (1e-5 is the tested bound). p(d) = t_d / S and the
 *     residual weights use it, so an acceptance whose |u - p(d)/q(d)|, or a residual race whose
 *     two best keys, lie within that margin may be decided differently from an implementation
 *     that sums S exactly; every other decision is reproducible bit for bit from these
 *     definitions.
 *   - sampled[i, :] holds the accepted drafts, then the recovered or bonus token, then -1.
 *     num_sampled[i] = accepted + 1, num_rejected[i] = K_i - accepted.
 *
 * Error behaviour: every entry point returns a status code (SV_OK or a negative SV_E*) and
 * never aborts the process. Problems visible on the host (NULL pointers, sizes beyond the
 * capacity given at init, dtype mismatch) are returned before anything is launched. Problems
 * in device data (cu_num_draft not starting at 0, decreasing, a K_i above
 * max_spec_len_this_batch, or a total different from num_draft_tokens) make every request of
 * that call emit num_sampled = num_rejected = 0 and a row of -1, and set SV_ERR_BATCH in the
 * context's error word (read with spec_verify_last_error).
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define SV_OK 0
#define SV_EINVAL (-1)    /* NULL or misaligned pointer, negative size, bad argument */
#define SV_ECAPACITY (-2) /* a size above the capacity given to spec_verify_init */
#define SV_EDTYPE (-3)    /* logits dtype not SV_F32 / SV_BF16 */
#define SV_ECUDA (-4)     /* a CUDA runtime call failed */
#define SV_EDEVICE (-5)   /* no usable device, or not an sm_103 device */

/* logits element types */
#define SV_F32 0  /* IEEE binary32 */
#define SV_BF16 1 /* bfloat16 (upper half of a binary32) */

/* draft inputs a context accepts (bits of spec_verify_init's draft_input) */
#define SV_DRAFT_PROBS 1  /* draft_probs may be given to spec_verify_run */
#define SV_DRAFT_LOGITS 2 /* spec_verify_run_draft_logits may be called */

/* most draft positions a synthetic acceptance setting can name */
#define SV_MAX_SYNTHETIC 64

/* bits of the device error word */
#define SV_ERR_BATCH 1u   /* inconsistent cu_num_draft / draft lengths in some call */
#define SV_ERR_COUNTS 2u  /* a counts_row outside [0, counts_rows): that request got no penalty */
#define SV_ERR_BOUNDS 4u  /* (a library built with SV_DEBUG_BOUNDS only) a kernel tried to read or
                             write outside the arrays of the call; the access was skipped */
#define SV_ERR_SELECT 8u  /* the top-k / top-p threshold of some row was not found within the
                             selection's pass limit (not expected to happen): that row was
                             left without the constraint */

typedef struct spec_verify_ctx spec_verify_ctx; /* opaque */

/*
 * Create a context on `device` (a CUDA ordinal) for batches of at most max_num_reqs requests,
 * at most max_spec_len draft tokens each, vocabulary size vocab_size and logits of type
 * logits_dtype (SV_F32 / SV_BF16). draft_input is 0 or an OR of SV_DRAFT_PROBS and
 * SV_DRAFT_LOGITS: without SV_DRAFT_PROBS draft_probs must always be NULL (only the
 * host-buffer entry point sizes anything by it); SV_DRAFT_LOGITS reserves the partial
 * statistics of the draft rows (about 16 * 8 * (vocab_size / 2048 + 2) bytes per draft row of
 * capacity) that spec_verify_run_draft_logits needs. Any other value returns SV_EINVAL.
 * The context owns its device scratch (the per-segment partial statistics, the frequency
 * penalty's counts mask of 4 * max_num_reqs * (ceil(vocab_size / 32) + 1) bytes, and an error
 * word), allocated here once; spec_verify_run allocates nothing. Free with spec_verify_free.
 * Returns SV_ECAPACITY when the race's per-group bounds of one row (about 12 bytes per 64
 * tokens) do not fit in one CTA's shared memory (vocab_size above about a million), and for
 * vocab_size >= 2^30.
 * Returns SV_OK and *out, or an error with *out = NULL.
 */
int spec_verify_init(spec_verify_ctx **out, int max_num_reqs, int max_spec_len, int vocab_size,
                     int logits_dtype, int draft_input, int device);

/*
 * Verify one batch, asynchronously on `cuda_stream` (a cudaStream_t; NULL = legacy default
 * stream). All pointers are device pointers owned by the caller and must stay valid until the
 * stream reaches the end of this call; logits and draft_probs must be 16-byte aligned.
 *   logits        [num_draft_tokens + num_reqs, vocab_size] of the context's dtype (layout above)
 *   draft_ids     [num_draft_tokens] int32
 *   draft_probs   [num_draft_tokens, vocab_size] binary32 distributions, or NULL (draft ids only)
 *   cu_num_draft  [num_reqs + 1] int32 prefix sums of the draft lengths, cu_num_draft[0] = 0
 *   temperature   [num_reqs] binary32;  is_greedy [num_reqs] uint8
 *   seed, req_index_base: RNG key and the request index of the first request (so a batch split
 *                 across calls or devices draws the same numbers as the whole batch)
 *   max_spec_len_this_batch: row length - 1 of `sampled`; every K_i must be <= it
 *   sampled       [num_reqs, max_spec_len_this_batch + 1] int32 (out)
 *   num_sampled, num_rejected  [num_reqs] int32 (out)
 *   opt_row_max, opt_row_sumexp [num_draft_tokens + num_reqs] binary32, opt_row_argmax int32:
 *                 optional (NULL to skip) per-row m = max_v x_v, S = sum_v exp(x_v - m) and the
 *                 raw-logit argmax, for every row including rows after a rejection (greedy rows
 *                 use T = 1 for m and S); not written when the batch is inconsistent.
 * The call performs no allocation and no host synchronisation and may be captured in a CUDA
 * graph. Calls on one context must not overlap on the device (they share its scratch).
 */
int spec_verify_run(spec_verify_ctx *ctx, const void *logits, const int32_t *draft_ids,
                    const float *draft_probs, const int32_t *cu_num_draft,
                    const float *temperature, const uint8_t *is_greedy, uint64_t seed,
                    uint32_t req_index_base, int num_reqs, int num_draft_tokens,
                    int max_spec_len_this_batch, int32_t *sampled, int32_t *num_sampled,
                    int32_t *num_rejected, float *opt_row_max, float *opt_row_sumexp,
                    int32_t *opt_row_argmax, void *cuda_stream);

/*
 * Probabilistic drafting with the draft model's logits instead of its probabilities
 * ([spec-in-vllm] 7.1: the probabilistic draft method keeps the full draft logits, one row of
 * V per draft step; 7.4: the statistics kernel reduces the draft logits as well as the
 * target's). q is computed inside the call and never written out:
 *   q_v = exp(y_v - m_d) / S_d,  y_v = draft_logit_v * (1 / T),  m_d = max_v y_v,
 *   S_d = sum_v exp(y_v - m_d),
 * with the request's own temperature T (the draft samples with the same settings), exp the
 * library's binary32 exp and the quotient correctly rounded in binary32; S_d is summed in an
 * unspecified order (relative error far below 1e-5). Acceptance and the residual race then use
 * this q exactly as spec_verify_run uses draft_probs. Greedy requests ignore q.
 *   draft_logits  [num_draft_tokens, vocab_size] of the context's dtype, 16-byte aligned, row
 *                 cu_num_draft[i] + j for draft j of request i (the layout of draft_probs).
 * Every other argument, the outputs and the error behaviour are those of spec_verify_run.
 * Returns SV_EINVAL if the context was created without SV_DRAFT_LOGITS. Both logits arrays
 * are reduced by one statistics launch; the call stays allocation-free and graph-capturable.
 */
int spec_verify_run_draft_logits(spec_verify_ctx *ctx, const void *logits,
                                 const int32_t *draft_ids, const void *draft_logits,
                                 const int32_t *cu_num_draft, const float *temperature,
                                 const uint8_t *is_greedy, uint64_t seed,
                                 uint32_t req_index_base, int num_reqs, int num_draft_tokens,
                                 int max_spec_len_this_batch, int32_t *sampled,
                                 int32_t *num_sampled, int32_t *num_rejected, float *opt_row_max,
                                 float *opt_row_sumexp, int32_t *opt_row_argmax,
                                 void *cuda_stream);

/*
 * One batch with every per-call input in one struct (device pointers, as spec_verify_run).
 * Fields: the arguments of spec_verify_run of the same names, and
 *   draft_logits     [num_draft_tokens, vocab_size] or NULL: as spec_verify_run_draft_logits
 *                    (needs SV_DRAFT_LOGITS; draft_probs must then be NULL)
 *   partial_prefill  [num_reqs] uint8 or NULL: requests whose prompt is still being prefilled
 *                    in chunks. Such a request reports num_sampled = num_rejected = 0 and a
 *                    row of -1 ([MTP-eagle] get_num_sampled_and_rejected: the count correction
 *                    for chunked prefill); its row statistics are still written.
 *   frequency_penalty [num_reqs] binary32, output_bin_counts [counts_rows, vocab_size] int32,
 *                    counts_row [num_reqs] int32 or NULL (= request i): the frequency penalty
 *                    ([MTP-eagle] 其他 / 重复惩罚: logit -= penalty * output_bin_counts[req],
 *                    applied before the temperature and the softmax, [spec-notes] 8.2). At
 *                    position j of request i the count of token v is
 *                    c = output_bin_counts[counts_row[i], v] + #{k < j : draft_k == v} (the
 *                    drafts before j are output the target conditions on there), and the
 *                    processed logit is fma(-penalty, c, logit) (one rounding; c as a
 *                    binary32 value rounded to nearest, exact below 2^24) where
 *                    penalty != 0 and c != 0, the logit itself otherwise; x = processed / T.
 *                    Greedy requests take the argmax of the processed logits; row_max /
 *                    row_argmax report them. The draft logits are not penalised. Both
 *                    frequency_penalty and output_bin_counts NULL: no penalty; one of them NULL
 *                    or counts_rows < 1 with the other set: SV_EINVAL. A counts_row outside
 *                    [0, counts_rows) gives that request no penalty and sets SV_ERR_COUNTS.
 *   top_k [num_reqs] int32, top_p [num_reqs] binary32, each or NULL: sampling constraints
 *                    applied to the processed logits before the softmax ([spec-notes] 8.2
 *                    apply_sampling_constraints; [mini-sglang]: top_k < 1 means the whole
 *                    vocabulary, top_p at most 1 and taken as at least 1e-6). For a sampling
 *                    request, with x sorted from the largest, top-k (1 <= k < V) keeps every
 *                    token at least the k-th largest value (ties kept); top-p (P < 1) then keeps,
 *                    among those, every token whose strictly larger tokens hold less than P of
 *                    their mass exp(x - m). p' = p on the kept set, renormalised, replaces p in
 *                    the acceptance test, the residual and every draw; row_sumexp reports the
 *                    kept mass. top_k == 1 makes the request greedy; greedy requests ignore
 *                    both. The kept masses are summed in binary32 (hardware exp2), so a top-p
 *                    boundary within about 1e-6 of the total may fall either way. These calls
 *                    launch one more kernel; spec_verify_run_noalloc does not take them.
 *   fp64_gumbel      0, or nonzero to draw the race noise in binary64 ([spec-in-vllm] 7.3:
 *                    use_fp64_gumbel, the Gumbel noise generated in double precision). Every
 *                    race of the call (residual, without the rejected draft, bonus, non-spec
 *                    Gumbel-max, synthetic mode's draw) then uses binary64 clocks with 52-bit
 *                    uniforms and compares binary64 keys: the same group layout as above, the
 *                    head call (g, j, i', 32) giving W = (m + 1/2) / 2^52 with
 *                    m = word0 * 2^20 + (word1 >> 12) and the slot a = word 2 & 63, slot s != a
 *                    taking U_s from words (0, 1) (even s) or (2, 3) (odd s) of counter
 *                    (g, j, i', 33 + s / 2), clocks E_g = -log(W) / 64 and E_g + (-log U_s) in
 *                    binary64 (log: the same reduction and atanh series, to the term 2/19), key
 *                    (double) w_v / E_v. The largest clock is then 53 ln 2 = 36.7 instead of
 *                    24 ln 2 = 16.6, so the noise's tail is no longer cut short in the far
 *                    tail of p. Acceptance tests are unchanged. Costs binary64 arithmetic (a
 *                    slow unit on this part) for the few tokens whose keys are evaluated
 *                    exactly. Not offered by the vocabulary-shard or no-alloc entry points.
 */
typedef struct spec_verify_batch {
    const void *logits;
    const int32_t *draft_ids;
    const float *draft_probs;
    const void *draft_logits;
    const int32_t *cu_num_draft;
    const float *temperature;
    const uint8_t *is_greedy;
    const uint8_t *partial_prefill;
    const float *frequency_penalty;
    const int32_t *output_bin_counts;
    const int32_t *counts_row;
    const int32_t *top_k;
    const float *top_p;
    uint64_t seed;
    uint32_t req_index_base;
    int32_t num_reqs;
    int32_t num_draft_tokens;
    int32_t max_spec_len_this_batch;
    int32_t counts_rows;
    int32_t fp64_gumbel;
} spec_verify_batch;

/* Outputs of one batch (device pointers): sampled, num_sampled, num_rejected as in
 * spec_verify_run; row_max, row_sumexp, row_argmax optional (NULL to skip). */
typedef struct spec_verify_outputs {
    int32_t *sampled;
    int32_t *num_sampled;
    int32_t *num_rejected;
    float *row_max;
    float *row_sumexp;
    int32_t *row_argmax;
} spec_verify_outputs;

/*
 * Verify the batch described by *batch into *out on `cuda_stream`. Same behaviour, errors and
 * guarantees as spec_verify_run (allocation-free, graph-capturable); spec_verify_run and
 * spec_verify_run_draft_logits are this call with the extra fields NULL.
 */
int spec_verify_run_batch(spec_verify_ctx *ctx, const spec_verify_batch *batch,
                          const spec_verify_outputs *out, void *cuda_stream);

/*
 * Synthetic acceptance ([spec-in-vllm] 7.2 and 7.4: instead of the acceptance test, draft
 * position j is accepted with a preset rate). rates[0..n) are the UNCONDITIONAL acceptance
 * rates a_j of positions j (the probability that position j is reached and accepted), each in
 * [0, 1] and non-increasing; positions j >= n have rate 0. Draft j is accepted iff
 * 0 <= d < V and c_j >= u_j, c_j = a_j / a_{j-1} (binary32 division, a_{-1} = 1; 0 when
 * a_{j-1} = 0) and u_j the acceptance uniform of the conventions above. The token at the
 * first rejection, or the bonus token, is the target's own choice: the argmax for greedy
 * requests, a draw from p (the race over p, nothing excluded) otherwise. draft_probs and
 * draft_logits are not used in this mode. Applies to every later call on the context;
 * n = 0 turns it off. rates is a HOST array, copied. Returns SV_EINVAL for n outside
 * [0, SV_MAX_SYNTHETIC], a rate outside [0, 1] (or NaN) or an increasing pair.
 */
int spec_verify_set_synthetic(spec_verify_ctx *ctx, const float *rates, int n);

/*
 * Per-position rates for a target mean accepted length ([spec-in-vllm] 7.2: a length in
 * [1, num_spec + 1] is turned into minimum-variance per-position rates). With A = mean_length
 * - 1 accepted drafts on average, the integer-valued count with the least variance takes only
 * floor(A) and floor(A) + 1: rates[j] = 1 for j < floor(A), A - floor(A) at j = floor(A), 0
 * after. Writes rates[0..num_spec) (a host array). Returns SV_EINVAL if mean_length is outside
 * [1, num_spec + 1] or num_spec is outside [0, SV_MAX_SYNTHETIC]. Needs no context or device.
 */
int spec_verify_synthetic_rates(double mean_length, int num_spec, float *rates);

/*
 * Vocabulary-sharded verification: the logits arrive split by vocabulary over `world` ranks (a
 * tensor-parallel LM head), rank r holding columns [v0_r, v0_r + Vs_r) of every row, each v0 a
 * multiple of 64 (race-clock groups stay on one rank). Instead of gathering the rows, each rank
 * makes three calls around two all-gathers of small records (the caller's collective):
 *   1. spec_verify_shard_stats: the shard's statistics record of every logit row;
 *      all-gather them (rank-major: [world][rows]);
 *   2. spec_verify_shard_race: every rank combines the records in rank order (so all take the
 *      same acceptance decisions, [spec-notes] 8.2 / 8.3), then races its shard at the row of
 *      the first rejection with the combined maximum and sum and the global race clocks; one
 *      record per request; all-gather them ([world][num_reqs]);
 *   3. spec_verify_shard_finish: the largest key over the shards wins (the residual or
 *      exclusion race where some shard has a candidate, else the race over p), and the outputs
 *      are written as by spec_verify_run.
 * The result equals spec_verify_run on the whole rows (up to S, summed in another order). The
 * context is created for the SHARD: vocab_size = Vs. Calls 1 and 2 of a step use the same
 * context on the same stream (2 reads what 1 left in its scratch). All pointers are device
 * pointers; draft_probs is the shard's columns [num_draft_tokens, Vs] or NULL. The batch must be
 * consistent (cu_num_draft as for spec_verify_run); logits processors, draft logits and
 * synthetic acceptance are not offered here.
 */
typedef struct spec_verify_shard_stat {
    float max_logit;    /* largest logit of the shard's part of the row */
    float sumexp;       /* sum over it of exp((logit - max_logit) / T) (greedy: T = 1) */
    int32_t argmax;     /* global index of the first largest logit */
    float draft_logit;  /* the row's draft token's logit if this shard holds it, else NaN */
    float draft_prob;   /* its draft probability (1 without draft_probs) if held, else NaN */
    int32_t reserved;
} spec_verify_shard_stat;

typedef struct spec_verify_shard_key {
    int32_t jstar;          /* first rejected position (K if none), the same on every rank */
    int32_t token;          /* a greedy request's token, else -1 */
    float residual_key;     /* the shard's best key of the residual / exclusion race */
    int32_t residual_index; /* its global token, -1 if the shard has no candidate */
    float p_key;            /* the shard's best key of the race over p (the bonus; the fallback,
                               taken only where the shard's own residual is empty) */
    int32_t p_index;
} spec_verify_shard_key;

int spec_verify_shard_stats(spec_verify_ctx *ctx, const void *logits_shard, int v0,
                            const int32_t *draft_ids, const float *draft_probs_shard,
                            const int32_t *cu_num_draft, const float *temperature,
                            const uint8_t *is_greedy, int num_reqs, int num_draft_tokens,
                            int max_spec_len_this_batch, spec_verify_shard_stat *out,
                            void *cuda_stream);

int spec_verify_shard_race(spec_verify_ctx *ctx, const void *logits_shard, int v0, int vocab_size,
                           const spec_verify_shard_stat *all_stats, int world,
                           const int32_t *draft_ids, const float *draft_probs_shard,
                           const int32_t *cu_num_draft, const float *temperature,
                           const uint8_t *is_greedy, uint64_t seed, uint32_t req_index_base,
                           int num_reqs, int num_draft_tokens, int max_spec_len_this_batch,
                           spec_verify_shard_key *out, void *cuda_stream);

int spec_verify_shard_finish(spec_verify_ctx *ctx, const spec_verify_shard_key *all_races,
                             int world, const int32_t *draft_ids, const int32_t *cu_num_draft,
                             int num_reqs, int max_spec_len_this_batch, int32_t *sampled,
                             int32_t *num_sampled, int32_t *num_rejected, void *cuda_stream);

/*
 * Allocate device staging buffers sized for the context's capacity (logits, draft_probs if
 * SV_DRAFT_PROBS, and the small per-request arrays) so that spec_verify_run_host can be used.
 */
int spec_verify_reserve_host_io(spec_verify_ctx *ctx);

/*
 * Same as spec_verify_run but every pointer is a HOST pointer (page-locked memory gives
 * asynchronous copies; pageable memory works too). The logits and the small per-request arrays
 * are copied to the context's staging buffers, the batch is verified, and sampled / num_sampled /
 * num_rejected are copied back; the call returns after the stream has finished (the outputs are
 * ready). draft_probs, of which the verifier reads only the draft's entry per position and the
 * entries of the few vocabulary groups its race evaluates, is read in place over the host link
 * when it is page-locked (allocated or registered through CUDA), and copied otherwise.
 * Requires spec_verify_reserve_host_io.
 */
int spec_verify_run_host(spec_verify_ctx *ctx, const void *logits, const int32_t *draft_ids,
                         const float *draft_probs, const int32_t *cu_num_draft,
                         const float *temperature, const uint8_t *is_greedy, uint64_t seed,
                         uint32_t req_index_base, int num_reqs, int num_draft_tokens,
                         int max_spec_len_this_batch, int32_t *sampled, int32_t *num_sampled,
                         int32_t *num_rejected, void *cuda_stream);

/*
 * Read and clear the context's device error word (SV_ERR_* bits) into *err_word. Waits for
 * the device (synchronises the context's device).
 */
int spec_verify_last_error(spec_verify_ctx *ctx, uint32_t *err_word);

/*
 * Kernel timing. With enable != 0, each later call records CUDA events around its kernels on
 * the call's stream. spec_verify_get_profile waits for the recorded work and returns, per
 * kernel, the summed milliseconds in ms[0 .. SV_PROFILE_SLOTS): 0 = row statistics, 1 = verify
 * (acceptance, race and emit), 2 = the top-k / top-p selection (0 in calls without it); and the
 * number of timed calls in *calls, then resets the sums.
 */
#define SV_PROFILE_SLOTS 3
int spec_verify_set_profiling(spec_verify_ctx *ctx, int enable);
int spec_verify_get_profile(spec_verify_ctx *ctx, double *ms, int64_t *calls);

/* Launch-shape knob: elements per CTA of the statistics kernel (0 keeps the current value; -1
 * restores the default, automatic: the flattened logits split evenly over the fewest whole waves
 * of CTAs whose chunk is at most 2^19 elements, one wave when that fits). Values are rounded up
 * to a multiple of 512 and kept between 2048 and 2^19. Results do not depend on it (S, a sum, up
 * to rounding). */
int spec_verify_set_chunks(spec_verify_ctx *ctx, int stats_chunk);

/* Number of kernel launches one call makes for a non-empty batch without top_k / top_p and
 * without a frequency penalty (one more, the selection kernel, with top_k / top_p; one more, the
 * counts-mask pass, with a penalty). */
int spec_verify_launches_per_run(void);

/*
 * Verification without any allocation, for callers that cannot allocate device memory: code
 * that runs inside another framework's memory pool or a plugin's execute call, where
 * cudaMalloc is forbidden or would synchronise the device at a bad moment, or processes whose
 * device memory is fully reserved up front. This entry point has no counterpart on the pages:
 * it is the same verification as spec_verify_run (same arguments, same results, the logits
 * type and vocabulary size given directly instead of through a context), but its scratch
 * space is a fixed static array inside the library (about 9.4 MB on every device that loads
 * it, held until the process exits).
 *   Limits: vocab_size <= SV_NOALLOC_MAX_VOCAB, num_reqs <= SV_NOALLOC_MAX_REQS, and
 *   num_draft_tokens + num_reqs <= SV_NOALLOC_MAX_ROWS; larger batches return SV_ECAPACITY.
 * It runs on the current device. Its first call on a device (or the first call of
 * spec_verify_noalloc_last_error there) sets the device up, once: it checks that the device
 * is an sm_103 part, looks up the array's device address and sets the kernels' shared-memory
 * limits; make that first call before any stream capture. Later calls on the device make no
 * CUDA runtime query besides the launches. All calls on a device share the array, so calls
 * that overlap on the GPU (different streams, or different host threads) race with each other
 * and must be serialised by the caller. An inconsistent cu_num_draft makes every request emit
 * num_sampled = num_rejected = 0 and a row of -1 and sets SV_ERR_BATCH in the array's error
 * word, which spec_verify_noalloc_last_error reads and clears. The frequency penalty, top-k /
 * top-p, draft logits and synthetic acceptance are not offered here.
 */
#define SV_NOALLOC_MAX_REQS 1024
#define SV_NOALLOC_MAX_ROWS 8192
#define SV_NOALLOC_MAX_VOCAB 262144
int spec_verify_run_noalloc(const void *logits, int logits_dtype, int vocab_size,
                            const int32_t *draft_ids, const float *draft_probs,
                            const int32_t *cu_num_draft, const float *temperature,
                            const uint8_t *is_greedy, uint64_t seed, uint32_t req_index_base,
                            int num_reqs, int num_draft_tokens, int max_spec_len_this_batch,
                            int32_t *sampled, int32_t *num_sampled, int32_t *num_rejected,
                            float *opt_row_max, float *opt_row_sumexp, int32_t *opt_row_argmax,
                            void *cuda_stream);

/*
 * Read and clear the error word of spec_verify_run_noalloc on the current device (SV_ERR_*
 * bits of every call since the last read), into *err_word. Like spec_verify_last_error it
 * waits for the device (synchronises it), so call it outside any stream capture. Allocates
 * nothing. Has no counterpart on the pages.
 */
int spec_verify_noalloc_last_error(uint32_t *err_word);

/* Release the context and its device memory. NULL is a no-op. */
void spec_verify_free(spec_verify_ctx *ctx);

/* Static description of a status code. */
const char *spec_verify_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
