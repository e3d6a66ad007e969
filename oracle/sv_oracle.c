/*
 * ORACLE FOR THE SPECULATIVE-DECODING VERIFICATION SAMPLER -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU restatement of what the verification step computes,
 * written from the pages' description. Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg use it; the library's product path never links, loads or calls it, and
 * it shares no code with the CUDA implementation.
 *
 * Pages cited (title, section):
 *   [MTP-eagle]     "【vllm】DeepSeekMTP、eagle" (benyoew.github.io): the sample() call tree,
 *                   _rejection_sample_kernel, get_num_sampled_and_rejected.
 *   [spec-notes]    "vLLM 投机解码（Eagle / MTP）实现与运行流程" (llx-08 notes): residual
 *                   distribution Q&A, bonus token and NO_DRAFT_PROBS Q&A, 4-token examples,
 *                   section 8 (rejection sampling) 8.2 / 8.3, section 9.2.
 *   [spec-in-vllm]  "speculative decoding in vLLM" (jiangwei.me): section 7.0 (5-token
 *                   example), 7.0.1 (greedy), 7.0.2 (bonus), 7.3 (Gumbel argmax), 7.4 (kernels).
 *   [mini-sglang]   "mini-sglang" (blog.thunguo.space): "how tokens are sampled" (greedy rule).
 *
 * Readings where the pages leave a step open:
 *   - p = softmax(logits / T) with x_v = logit_v * (1/T) in binary32; T <= 0 (or a set greedy
 *     flag) means greedy verification.
 *   - Acceptance test p(d)/q(d) >= u with u in (0,1); q(d) = 1 without draft probabilities.
 *   - Every random draw is keyed: Philox4x32-10, key = seed, counter words (c0, j, request,
 *     c3). The acceptance uniform of position j is word 0 of counter (0, j, request, 0).
 *   - Sampling from a distribution proportional to w_v is the exponential race
 *     argmax_v w_v / E_v over i.i.d. Exp(1) clocks E_v (the key is the binary32 quotient),
 *     lowest index on equal keys; over p the weight is t_v = exp(x_v - m).
 *     The clocks come in groups of 64 tokens (group g = v >> 6, slot s = v & 63): counter
 *     (g, j, request, 8) gives W (word 0) and the slot a = word 1 & 63 holding the group's
 *     smallest clock E_min = -log(W) / 64; the other slots' clocks are E_min + (-log U_s), U_s
 *     word s & 3 of counter (g, j, request, 9 + s / 4). By the memoryless property of the
 *     exponential these 64 clocks are i.i.d. Exp(1).
 *   - The residual weight is rr_v = fma(-S, q_v, t_v) with t_v = exp(x_v - m), i.e.
 *     S * (p_v - q_v) rounded once; the constant factor 1 / S is left out of the keys.
 *   - exp and log inside every decision are the binary32 functions below (Cody-Waite
 *     reduction + Taylor polynomial; reduction to [sqrt(1/2), sqrt(2)) + atanh series), so
 *     that any implementation that follows the same steps gets the same bits.
 *   - S, the sum of exponentials, is accumulated in double in index order.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define REF_TAG_ACCEPT 0u  /* counter word 3 of the acceptance uniform */
#define REF_CLOCK_HEAD 8u  /* counter word 3 of a group's head call; its slot calls use 9..24 */

/* ------------------------------------------------------------------------------------ */
/* Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
 * SC'11. Each round multiplies counter words 0 and 2 by the round multipliers, and the
 * key is bumped by the Weyl constants (golden ratio, sqrt(3)-1) between rounds.         */
/* ------------------------------------------------------------------------------------ */
void spec_verify_ref_philox(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    const uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)M0 * c0;
        uint64_t p1 = (uint64_t)M1 * c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        k0 += W0;
        k1 += W1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Uniform in (0,1): the top 23 bits of a Philox word w, centred in their cell,
 * U = (floor(w / 2^9) + 1/2) / 2^23. Every step is exact in binary32, U is never 0 or 1. */
float spec_verify_ref_uniform_from_word(uint32_t w)
{
    return ((float)(w >> 9) + 0.5f) * 0x1p-23f;
}

float spec_verify_ref_uniform(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                              int word)
{
    uint32_t ctr[4] = {c0, c1, c2, c3};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    spec_verify_ref_philox(ctr, key, out);
    return spec_verify_ref_uniform_from_word(out[word & 3]);
}

/* ------------------------------------------------------------------------------------ */
/* binary32 exp and log used inside every decision.                                      */
/* ------------------------------------------------------------------------------------ */
static inline float bits_f(uint32_t b) { float f; memcpy(&f, &b, 4); return f; }
static inline uint32_t f_bits(float f) { uint32_t b; memcpy(&b, &f, 4); return b; }

#define REF_LOG2E 0x1.715476p+0f   /* log2(e) rounded to binary32 */
#define REF_LN2_HI 0x1.62e430p-1f  /* ln 2 rounded to binary32 */
#define REF_LN2_LO -0x1.05c610p-29f /* ln 2 - REF_LN2_HI, rounded to binary32 */

/* exp(d) for d <= 88, defined as 0 below -87 (where exp(d) < 1.7e-38).
 * Cody & Waite (1980) reduction d = k ln2 + r, |r| <= ln2/2, with k = round(d log2 e) taken
 * by adding 1.5*2^23 in one fused multiply-add; exp(r) by its Taylor polynomial of degree 7
 * (truncation error < 6e-9 relative) in Horner form; the result is exp(r) * 2^k. */
float spec_verify_ref_exp(float d)
{
    if (!(d >= -87.0f)) return d != d ? d : 0.0f;
    if (d > 88.0f) return INFINITY;
    const float shifter = 0x1.8p+23f;
    float kf = fmaf(d, REF_LOG2E, shifter) - shifter;
    float r = fmaf(-kf, REF_LN2_HI, d);
    r = fmaf(-kf, REF_LN2_LO, r);
    float p = 0x1.a01a02p-13f;            /* 1/7! */
    p = fmaf(p, r, 0x1.6c16c2p-10f);      /* 1/6! */
    p = fmaf(p, r, 0x1.111112p-7f);       /* 1/5! */
    p = fmaf(p, r, 0x1.555556p-5f);       /* 1/4! */
    p = fmaf(p, r, 0x1.555556p-3f);       /* 1/3! */
    p = fmaf(p, r, 0.5f);                 /* 1/2! */
    p = fmaf(p, r, 1.0f);
    p = fmaf(p, r, 1.0f);
    int k = (int)kf;
    return p * bits_f((uint32_t)(k + 127) << 23);
}

/* log(x) for finite x > 0 (0 -> -inf, negative or NaN -> NaN, +inf -> +inf).
 * x = 2^k f with f in [sqrt(1/2), sqrt(2)); ln f = 2 atanh(s), s = (f-1)/(f+1), |s| < 0.172,
 * summed as 2s + s z (2/3 + z (2/5 + z (2/7 + z 2/9))), z = s^2 (truncation < 1e-9
 * relative); ln x = k ln2 + ln f. Subnormal x is scaled by 2^23 first. */
float spec_verify_ref_log(float x)
{
    if (x != x || x < 0.0f) return NAN;
    if (x == 0.0f) return -INFINITY;
    if (x == INFINITY) return INFINITY;
    int k = 0;
    uint32_t b = f_bits(x);
    if (b < 0x00800000u) {
        b = f_bits(x * 0x1p+23f);
        k = -23;
    }
    k += (int)(b >> 23) - 127;
    uint32_t fb = (b & 0x007FFFFFu) | 0x3F800000u;
    if (fb > 0x3FB504F3u) { /* f > sqrt(2): halve it */
        fb -= 0x00800000u;
        k += 1;
    }
    float f = bits_f(fb);
    float g = f - 1.0f;
    float s = g / (g + 2.0f);
    float z = s * s;
    float P = fmaf(z, 0x1.c71c72p-3f, 0x1.24924ap-2f); /* 2/9, 2/7 */
    P = fmaf(z, P, 0x1.99999ap-2f);                    /* 2/5 */
    P = fmaf(z, P, 0x1.555556p-1f);                    /* 2/3 */
    float R = z * P;
    float lnf = fmaf(s, R, s + s);
    float kf = (float)k;
    return fmaf(kf, REF_LN2_HI, fmaf(kf, REF_LN2_LO, lnf));
}

/* Race clock of token v at position j of request ireq (see the header): i.i.d. Exp(1). */
float spec_verify_ref_race_clock(uint64_t seed, uint32_t j, uint32_t ireq, int32_t v)
{
    const uint32_t g = (uint32_t)v >> 6;
    const uint32_t slot = (uint32_t)v & 63u;
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {g, j, ireq, REF_CLOCK_HEAD};
    uint32_t head[4];
    spec_verify_ref_philox(ctr, key, head);
    const float W = spec_verify_ref_uniform_from_word(head[0]);
    const uint32_t a = head[1] & 63u;
    const float emin = -spec_verify_ref_log(W) * 0.015625f; /* E_W / 64, exact scaling */
    if (slot == a) return emin;
    ctr[3] = REF_CLOCK_HEAD + 1u + slot / 4u;
    uint32_t words[4];
    spec_verify_ref_philox(ctr, key, words);
    const float U = spec_verify_ref_uniform_from_word(words[slot & 3u]);
    return emin + (-spec_verify_ref_log(U));
}

/* ------------------------------------------------------------------------------------ */
/* Race clocks drawn in binary64 ([spec-in-vllm] 7.3: use_fp64_gumbel, the race noise      */
/* generated in double precision). Same layout idea as the binary32 clocks, 52-bit          */
/* uniforms from two Philox words each, a separate counter range (word 3 = 32 .. 64).      */
/* ------------------------------------------------------------------------------------ */
#define REF_CLOCK_HEAD64 32u /* counter word 3 of a group's binary64 head call; slots use 33..64 */

static inline double bits_d(uint64_t b) { double d; memcpy(&d, &b, 8); return d; }
static inline uint64_t d_bits(double d) { uint64_t b; memcpy(&b, &d, 8); return b; }

/* Uniform in (0,1) from two Philox words: the top 52 bits of (hi, lo), centred in their cell,
 * U = (m + 1/2) / 2^52 with m = hi * 2^20 + (lo >> 12). m + 1/2 has 53 significant bits, so
 * every step is exact in binary64; U lies in [2^-53, 1 - 2^-53]. */
double spec_verify_ref_uniform64(uint32_t hi, uint32_t lo)
{
    const uint64_t m = ((uint64_t)hi << 20) | (uint64_t)(lo >> 12);
    return ((double)m + 0.5) * 0x1p-52;
}

#define REF_LN2_HI64 0x1.62e42fefa3800p-1  /* ln 2 rounded to 42 significant bits: k ln2_hi exact */
#define REF_LN2_LO64 0x1.ef35793c76730p-45 /* ln 2 - REF_LN2_HI64, rounded to binary64 */

/* binary64 log for x > 0, the same method as the binary32 log: x = 2^k f with f in
 * [sqrt(1/2), sqrt(2)), ln f = 2 atanh(s), s = (f - 1) / (f + 1), |s| < 0.1716, summed as
 * 2s + s z P(z), z = s^2, P(z) = 2/3 + z (2/5 + z (... + z 2/19)) (the terms 2 s^(2n+1)/(2n+1)
 * up to n = 9; the first one left out, 2 s^21 / 21, is below 0.15 ulp of the result); ln x =
 * k ln 2 + ln f with the two-part ln 2 above. Subnormals are scaled by 2^54 first. 0 -> -inf,
 * negative or NaN -> NaN, +inf -> +inf. */
double spec_verify_ref_log64(double x)
{
    if (x != x || x < 0.0) return NAN;
    if (x == 0.0) return -INFINITY;
    if (x == INFINITY) return INFINITY;
    int k = 0;
    uint64_t b = d_bits(x);
    if (b < 0x0010000000000000ull) {
        b = d_bits(x * 0x1p+54);
        k = -54;
    }
    k += (int)(b >> 52) - 1023;
    uint64_t fb = (b & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull;
    if (fb > 0x3FF6A09E667F3BCCull) { /* f > sqrt(2) (the largest double below it is ...BCC) */
        fb -= 0x0010000000000000ull;
        k += 1;
    }
    const double f = bits_d(fb);
    const double g = f - 1.0;
    const double s = g / (g + 2.0);
    const double z = s * s;
    double P = fma(z, 0x1.af286bca1af28p-4, 0x1.e1e1e1e1e1e1ep-4); /* 2/19, 2/17 */
    P = fma(z, P, 0x1.1111111111111p-3);                          /* 2/15 */
    P = fma(z, P, 0x1.3b13b13b13b14p-3);                          /* 2/13 */
    P = fma(z, P, 0x1.745d1745d1746p-3);                          /* 2/11 */
    P = fma(z, P, 0x1.c71c71c71c71cp-3);                          /* 2/9 */
    P = fma(z, P, 0x1.2492492492492p-2);                          /* 2/7 */
    P = fma(z, P, 0x1.999999999999ap-2);                          /* 2/5 */
    P = fma(z, P, 0x1.5555555555555p-1);                          /* 2/3 */
    const double R = z * P;
    const double lnf = fma(s, R, s + s);
    const double kf = (double)k;
    return fma(kf, REF_LN2_HI64, fma(kf, REF_LN2_LO64, lnf));
}

/* Race clock of token v at position j of request ireq, drawn in binary64: group g = v >> 6,
 * slot s = v & 63; counter (g, j, ireq, 32) gives W = uniform64(word 0, word 1) and the slot
 * a = word 2 & 63 holding the group's smallest clock E_min = -log(W) / 64; slot s != a has
 * clock E_min + (-log U_s), U_s = uniform64 of words (0, 1) (s even) or (2, 3) (s odd) of
 * counter (g, j, ireq, 33 + s / 2). By the memoryless property the 64 clocks are i.i.d.
 * Exp(1), as in binary32, with 52-bit instead of 23-bit uniforms (the largest clock is
 * 53 ln 2 = 36.7 instead of 24 ln 2 = 16.6). */
double spec_verify_ref_race_clock64(uint64_t seed, uint32_t j, uint32_t ireq, int32_t v)
{
    const uint32_t g = (uint32_t)v >> 6;
    const uint32_t slot = (uint32_t)v & 63u;
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t ctr[4] = {g, j, ireq, REF_CLOCK_HEAD64};
    uint32_t head[4];
    spec_verify_ref_philox(ctr, key, head);
    const double W = spec_verify_ref_uniform64(head[0], head[1]);
    const uint32_t a = head[2] & 63u;
    const double emin = -spec_verify_ref_log64(W) * 0x1p-6; /* exact scaling */
    if (slot == a) return emin;
    ctr[3] = REF_CLOCK_HEAD64 + 1u + slot / 2u;
    uint32_t words[4];
    spec_verify_ref_philox(ctr, key, words);
    const int h = (slot & 1u) ? 2 : 0;
    const double U = spec_verify_ref_uniform64(words[h], words[h + 1]);
    return emin + (-spec_verify_ref_log64(U));
}

/* ------------------------------------------------------------------------------------ */
/* The verification step.                                                                */
/* ------------------------------------------------------------------------------------ */
enum { REF_OK = 0, REF_EINVAL = -1, REF_EBATCH = 1 };
enum { REF_RACE_NONE = 0, REF_RACE_RESIDUAL = 1, REF_RACE_EXCLUDE = 2, REF_RACE_BONUS = 3,
       REF_RACE_FALLBACK = 4, REF_RACE_TARGET = 5 };

/* Options of a verification call (NULL pointer = all off).
 *   synthetic_rates: synthetic acceptance ([spec-in-vllm] 7.2): the unconditional acceptance
 *       rate a_j of draft positions j < num_synthetic_rates (a_j = 0 beyond), in [0, 1] and
 *       non-increasing. Replaces every request's acceptance test (7.4: the rejection kernel
 *       compares with the preset rate in this mode).
 *   partial_prefill: [num_reqs] or NULL; a request still in a chunked prefill reports no
 *       token ([MTP-eagle] get_num_sampled_and_rejected: the count correction for chunked
 *       prefill).
 *   frequency_penalty [num_reqs], output_bin_counts [counts_rows x V] with counts_row
 *       [num_reqs] (the counts row of each request; NULL = row i): the frequency penalty (see
 *       processed_row). Either pointer NULL: no penalty; a counts row outside
 *       [0, counts_rows): no penalty for that request.
 *   top_k [num_reqs] int32, top_p [num_reqs] binary32, each or NULL: sampling constraints of
 *       sampling requests (see select_row). top_k == 1 makes a request greedy.
 *   row_select_margin [rows] (output, NULL to skip): the top-p decision margin of each row.
 *   fp64_gumbel: nonzero draws every race's clocks in binary64 (spec_verify_ref_race_clock64)
 *       and compares its keys w_v / E_v as binary64 quotients ([spec-in-vllm] 7.3
 *       use_fp64_gumbel); the acceptance uniforms are unchanged. */
typedef struct {
    const float *synthetic_rates;
    int32_t num_synthetic_rates;
    const uint8_t *partial_prefill;
    const float *frequency_penalty;
    const int32_t *output_bin_counts;
    const int32_t *counts_row;
    int32_t counts_rows;
    const int32_t *top_k;
    const float *top_p;
    double *row_select_margin;
    int32_t fp64_gumbel;
} ref_options_t;

/* Conditional acceptance probability of position j given that positions 0..j-1 were
 * accepted: a_j / a_{j-1} (a_{-1} = 1), so that position j is reached and accepted with
 * probability a_j. A position that cannot be reached (a_{j-1} = 0) gets 0. */
static float synthetic_conditional(const ref_options_t *o, int j)
{
    const float a = j < o->num_synthetic_rates ? o->synthetic_rates[j] : 0.0f;
    if (j == 0) return a;
    const float prev = j - 1 < o->num_synthetic_rates ? o->synthetic_rates[j - 1] : 0.0f;
    return prev > 0.0f ? a / prev : 0.0f;
}

/* Per-position rates for a target mean accepted length L in [1, num_spec + 1]
 * ([spec-in-vllm] 7.2: the length is turned into minimum-variance per-position rates).
 * The number of accepted drafts N has mean L - 1; among laws of an integer N with that mean the
 * variance is smallest when N takes only floor(L - 1) and floor(L - 1) + 1, so
 * a_j = P(N > j) = 1 for j < floor(L - 1), the fractional part of L - 1 at j = floor(L - 1),
 * and 0 after. Returns REF_EINVAL if L is out of range. */
int spec_verify_ref_synthetic_rates(double mean_length, int num_spec, float *rates)
{
    if (num_spec < 0 || !(mean_length >= 1.0 && mean_length <= num_spec + 1.0)) return REF_EINVAL;
    const double a = mean_length - 1.0;
    const int n = (int)floor(a);
    for (int j = 0; j < num_spec; ++j)
        rates[j] = j < n ? 1.0f : (j == n ? (float)(a - n) : 0.0f);
    return REF_OK;
}

static inline float logit_at(const void *logits, int bf16, size_t idx)
{
    if (bf16) return bits_f((uint32_t)((const uint16_t *)logits)[idx] << 16);
    return ((const float *)logits)[idx];
}

/* Processed logits of one row ([spec-notes] 8.2: the logits processors run before the
 * softmax):
 *   y_v = fma(-f, c_v, l_v)  ([MTP-eagle] frequency penalty: logit -= penalty * count), and
 *   y_v = l_v where f = 0 or c_v = 0;
 *   x_v = y_v * (1 / T).
 * c_v is the token's count in `counts` (none without counts) plus the number of drafts before
 * this position that equal v: the drafts before position j are output the target conditions
 * on at j. */
static void processed_row(const void *logits, int bf16, size_t row, int V, float invT, float f,
                          const int32_t *counts, const int32_t *prev, int nprev, float *y, float *x)
{
    const size_t base = row * (size_t)V;
    for (int v = 0; v < V; ++v) {
        const float l = logit_at(logits, bf16, base + (size_t)v);
        int64_t c = counts ? counts[v] : 0;
        for (int k = 0; k < nprev; ++k) c += prev[k] == v;
        y[v] = (f == 0.0f || c == 0) ? l : fmaf(-f, (float)c, l);
        x[v] = y[v] * invT;
    }
}

typedef struct {
    float m;       /* max_v x_v */
    double S;      /* sum_v exp(x_v - m), accumulated in double in index order */
    float S_f;     /* S rounded to binary32 */
    int32_t amax;  /* argmax of y (the processed logits before temperature), lowest index */
    float tau;     /* kept tokens: x_v >= tau (-inf: all) */
    double Sk;     /* sum over the kept tokens of exp(x_v - m), double, index order */
    float Sk_f;    /* Sk rounded to binary32: the normaliser of p' that the decisions use */
    double margin; /* top-p decision margin relative to its total (+inf without top-p) */
} row_stats_t;

/* Softmax statistics of one processed row: [spec-in-vllm] 7.4 (block stats: max, argmax, sum
 * of exp, for a log-sum-exp) and [spec-notes] 8.2 (target probs = softmax of the processed
 * logits). */
static row_stats_t row_stats(const float *y, const float *x, int V)
{
    row_stats_t st;
    st.m = -INFINITY;
    st.amax = 0;
    for (int v = 0; v < V; ++v) {
        if (x[v] > st.m) st.m = x[v];
        if (y[v] > y[st.amax]) st.amax = v;
    }
    double S = 0.0;
    for (int v = 0; v < V; ++v) S += (double)spec_verify_ref_exp(x[v] - st.m);
    st.S = S;
    st.S_f = (float)S;
    st.tau = -INFINITY;
    st.Sk = S;
    st.Sk_f = st.S_f;
    st.margin = INFINITY;
    return st;
}

typedef struct {
    float x;
    int32_t v;
} xv_t;

static int by_value_desc(const void *a, const void *b)
{
    const xv_t *p = (const xv_t *)a, *q = (const xv_t *)b;
    if (p->x != q->x) return p->x > q->x ? -1 : 1;
    return p->v < q->v ? -1 : (p->v > q->v);
}

/* Sampling constraints ([spec-notes] 8.2 apply_sampling_constraints; [mini-sglang]: top_k < 1
 * means the whole vocabulary, top_p is clamped to [1e-6, 1]). With the values sorted from the
 * largest:
 *   top-k keeps every token whose value is at least the k-th largest (ties at the boundary are
 *         all kept), for 1 <= k < V;
 *   top-p then keeps, among those, every token whose strictly larger tokens hold less than
 *         P * Z of the mass, Z the mass of the top-k set (mass t_v = exp(x_v - m), summed in
 *         double), for P < 1.
 * Both keep a set {x_v >= tau}; p' is p restricted to it and renormalised by Sk. */
static void select_row(const float *x, int V, int top_k, float top_p, row_stats_t *st)
{
    const int use_k = top_k >= 1 && top_k < V;
    const int use_p = top_p < 1.0f; /* NaN or >= 1: no top-p */
    if (!use_k && !use_p) return;
    const double P = top_p < 1e-6f ? 1e-6 : (double)top_p;
    xv_t *s = (xv_t *)malloc((size_t)V * sizeof(xv_t));
    for (int v = 0; v < V; ++v) {
        s[v].x = x[v];
        s[v].v = v;
    }
    qsort(s, (size_t)V, sizeof(xv_t), by_value_desc);
    const float tau_k = use_k ? s[top_k - 1].x : -INFINITY;
    double Z = 0.0;
    for (int v = 0; v < V; ++v)
        if (x[v] >= tau_k) Z += (double)spec_verify_ref_exp(x[v] - st->m);
    float tau = tau_k;
    double margin = INFINITY;
    if (use_p) {
        const double target = P * Z;
        double above = 0.0; /* mass of the tokens strictly larger than the current group */
        int k = 0;
        while (k < V && s[k].x >= tau_k) {
            const float xv = s[k].x;
            double gm = 0.0;
            int e = k;
            for (; e < V && s[e].x == xv; ++e) gm += (double)spec_verify_ref_exp(xv - st->m);
            if (above < target) {
                tau = xv;
                if ((target - above) / Z < margin) margin = (target - above) / Z;
                above += gm;
                k = e;
            } else {
                if ((above - target) / Z < margin) margin = (above - target) / Z;
                break;
            }
        }
    }
    free(s);
    double Sk = 0.0;
    for (int v = 0; v < V; ++v)
        if (x[v] >= tau) Sk += (double)spec_verify_ref_exp(x[v] - st->m);
    st->tau = tau;
    st->Sk = Sk;
    st->Sk_f = (float)Sk;
    st->margin = margin;
}

typedef struct {
    int32_t idx;   /* winner, or -1 when no candidate */
    double key;    /* winner's key (a binary32 value unless the clocks are binary64) */
    double gap;    /* winner's key minus the runner-up's (+inf with fewer than two) */
    int64_t ncand; /* number of candidates */
} race_t;

/* Offer candidate v (offered in increasing v): the larger key wins, and an equal key at a
 * higher index loses to the earlier one, so the winner is the lowest index among the largest
 * keys. `second` tracks the runner-up key for the decision margin. */
static inline void race_offer(race_t *r, double key, int32_t v, double *second)
{
    r->ncand++;
    if (r->idx < 0) {
        r->key = key;
        r->idx = v;
    } else if (key > r->key) {
        *second = r->key;
        r->key = key;
        r->idx = v;
    } else if (key > *second) {
        *second = key;
    }
}

/* Exponential race over one row at position j of request ireq, [spec-notes] NO_DRAFT_PROBS
 * answer (argmax(prob / q) with q ~ Exp(1) needs no normalisation) and [spec-in-vllm] 7.3
 * (Gumbel argmax, the same race in log form). Keys: key_v = w_v / E_v, E_v the token's race
 * clock, one binary32 division.
 * Only the tokens the sampling constraints keep (x_v >= tau) take part; S is the normaliser of
 * p over them.
 *   q == NULL : w_v = t_v = exp(x_v - m), proportional to p_v; token `exclude` is left out
 *               (the rejected draft token when there are no draft probabilities).
 *   q != NULL : residual weights rr_v = fma(-S, q_v, t_v) = S (p_v - q_v) rounded once,
 *               candidates rr_v > 0 ([spec-notes] residual distribution max(0, p - q)).
 * The decision margin is the winner's key over the runner-up's, as log(key1) - log(key2).
 * fp64: the clocks are binary64 (spec_verify_ref_race_clock64) and the key is the binary64
 * quotient (double) w_v / E_v.                                                              */
static race_t race_row(const float *x, int V, float m, float tau, float S_f, const float *q,
                       int32_t exclude, uint64_t seed, uint32_t j, uint32_t ireq, int fp64)
{
    race_t r = {-1, -INFINITY, INFINITY, 0};
    double second = -INFINITY;
    for (int v = 0; v < V; ++v) {
        if (v == exclude || !(x[v] >= tau)) continue; /* only kept tokens take part */
        float t = spec_verify_ref_exp(x[v] - m);
        float w;
        if (q) {
            float rr = fmaf(-S_f, q[v], t);
            if (!(rr > 0.0f)) continue;
            w = rr;
        } else {
            w = t;
        }
        double key;
        if (fp64) {
            key = (double)w / spec_verify_ref_race_clock64(seed, j, ireq, v);
        } else {
            const float E = spec_verify_ref_race_clock(seed, j, ireq, v);
            key = (double)(w / E); /* the binary32 quotient */
        }
        race_offer(&r, key, v, &second);
    }
    if (r.idx >= 0 && r.ncand >= 2)
        r.gap = second > 0.0 ? log(r.key) - log(second) : INFINITY;
    return r;
}

/*
 * Verify one batch. Layout ([MTP-eagle] sample(): num_draft + 1 logit rows per request):
 *   logits       [num_draft_tokens + num_reqs, V], row of (request i, position j) is
 *                cu_num_draft[i] + i + j, j = K_i is the bonus row; bf16 bits or binary32.
 *   draft_ids    [num_draft_tokens], draft j of request i at cu_num_draft[i] + j.
 *   draft_probs  [num_draft_tokens, V] binary32 or NULL (no draft probabilities).
 *   temperature, is_greedy [num_reqs].
 * Outputs: sampled [num_reqs, max_spec_len + 1] (-1 padded), num_sampled, num_rejected.
 * Optional diagnostics (NULL to skip): row_max, row_sumexp (binary32 S), row_argmax per row;
 * accept_margin per draft position (|u - p/q| in double; +inf for greedy or invalid ids;
 * NaN where not evaluated); race_gap, race_kind, jstar per request.
 * u_override (test hook, NULL normally): acceptance uniforms per draft position.
 * opts: synthetic acceptance and chunked-prefill flags (see ref_options_t), or NULL.
 * Returns 0; REF_EBATCH when cu_num_draft is inconsistent (then every request emits
 * num_sampled = num_rejected = 0 and a row of -1); REF_EINVAL for bad arguments.
 */
int spec_verify_ref_run(const void *logits, int logits_bf16, int vocab_size,
                        const int32_t *draft_ids, const float *draft_probs,
                        const int32_t *cu_num_draft, const float *temperature,
                        const uint8_t *is_greedy, uint64_t seed, uint32_t req_index_base,
                        int num_reqs, int num_draft_tokens, int max_spec_len, int32_t *sampled,
                        int32_t *num_sampled, int32_t *num_rejected, float *row_max,
                        float *row_sumexp, int32_t *row_argmax, double *accept_margin,
                        double *race_gap, int32_t *race_kind, int32_t *jstar_out,
                        const float *u_override, const ref_options_t *opts)
{
    if (num_reqs < 0 || num_draft_tokens < 0 || max_spec_len < 0 || vocab_size <= 0) return REF_EINVAL;
    const int V = vocab_size;
    const int stride = max_spec_len + 1;
    int bad = cu_num_draft[0] != 0 || cu_num_draft[num_reqs] != num_draft_tokens;
    for (int i = 0; i < num_reqs && !bad; ++i) {
        int K = cu_num_draft[i + 1] - cu_num_draft[i];
        bad = K < 0 || K > max_spec_len;
    }
    if (accept_margin)
        for (int k = 0; k < num_draft_tokens; ++k) accept_margin[k] = NAN;
    if (bad) {
        for (int i = 0; i < num_reqs; ++i) {
            for (int s = 0; s < stride; ++s) sampled[(size_t)i * stride + s] = -1;
            num_sampled[i] = 0;
            num_rejected[i] = 0;
            if (race_gap) race_gap[i] = INFINITY;
            if (race_kind) race_kind[i] = REF_RACE_NONE;
            if (jstar_out) jstar_out[i] = -1;
        }
        return REF_EBATCH;
    }

    for (int i = 0; i < num_reqs; ++i) {
        const int q0 = cu_num_draft[i];
        const int K = cu_num_draft[i + 1] - q0;
        const size_t row0 = (size_t)q0 + (size_t)i;
        const uint32_t ireq = req_index_base + (uint32_t)i;
        const float T = temperature[i];
        const int top_k = opts && opts->top_k ? opts->top_k[i] : 0;
        const float top_p = opts && opts->top_p ? opts->top_p[i] : 1.0f;
        /* greedy: flag set, or temperature 0 ([spec-in-vllm] 7.0.1; [mini-sglang] T <= 0, and
         * top_k == 1 keeps only the largest logit) */
        const int greedy = is_greedy[i] != 0 || !(T > 0.0f) || top_k == 1;
        const float invT = greedy ? 1.0f : 1.0f / T;
        const int32_t crow = opts && opts->counts_row ? opts->counts_row[i] : i;
        const int pen = opts && opts->frequency_penalty && opts->output_bin_counts && crow >= 0 &&
                        crow < opts->counts_rows;
        const float f = pen ? opts->frequency_penalty[i] : 0.0f;
        const int32_t *counts = pen ? opts->output_bin_counts + (size_t)crow * (size_t)V : NULL;

        /* processed logits and stats of every row (rows after a rejection are reported too,
         * for inspection); row j conditions on the drafts before it */
        float *ybuf = (float *)malloc((size_t)(K + 1) * V * sizeof(float));
        float *xbuf = (float *)malloc((size_t)(K + 1) * V * sizeof(float));
        row_stats_t st[K + 1];
        for (int j = 0; j <= K; ++j) {
            float *y = ybuf + (size_t)j * V, *x = xbuf + (size_t)j * V;
            processed_row(logits, logits_bf16, row0 + (size_t)j, V, invT, f, counts,
                          draft_ids + q0, pen ? j : 0, y, x);
            st[j] = row_stats(y, x, V);
            if (!greedy) select_row(x, V, top_k, top_p, &st[j]);
            if (row_max) row_max[row0 + j] = st[j].m;
            if (row_sumexp) row_sumexp[row0 + j] = st[j].Sk_f;
            if (row_argmax) row_argmax[row0 + j] = st[j].amax;
            if (opts && opts->row_select_margin) opts->row_select_margin[row0 + j] = st[j].margin;
        }

        /* a request still in its chunked prefill reports no token and no rejection */
        if (opts && opts->partial_prefill && opts->partial_prefill[i]) {
            for (int s = 0; s < stride; ++s) sampled[(size_t)i * stride + s] = -1;
            num_sampled[i] = 0;
            num_rejected[i] = 0;
            if (race_gap) race_gap[i] = INFINITY;
            if (race_kind) race_kind[i] = REF_RACE_NONE;
            if (jstar_out) jstar_out[i] = -1;
            free(ybuf);
            free(xbuf);
            continue;
        }
        const int synthetic = opts && opts->synthetic_rates;
        const int fp64 = opts && opts->fp64_gumbel;

        /* [MTP-eagle] _rejection_sample_kernel: walk the draft positions, stop at the
         * first rejection; [spec-notes] 8.3 greedy and stochastic rules. */
        int jstar = K;
        for (int j = 0; j < K; ++j) {
            const int32_t d = draft_ids[q0 + j];
            int acc;
            double margin;
            if (synthetic) {
                /* [spec-in-vllm] 7.2 / 7.4: accept with the preset rate, whatever the tokens */
                const float c = synthetic_conditional(opts, j);
                const float u = u_override
                                    ? u_override[q0 + j]
                                    : spec_verify_ref_uniform(seed, 0u, (uint32_t)j, ireq,
                                                              REF_TAG_ACCEPT, 0);
                acc = d >= 0 && d < V && c >= u; /* an invalid id is still rejected */
                margin = d >= 0 && d < V ? fabs((double)u - (double)c) : INFINITY;
            } else if (greedy) {
                acc = d == st[j].amax;
                margin = INFINITY;
            } else if (d < 0 || d >= V) {
                acc = 0; /* [spec-notes] accept only when draft_token_id < vocab_size */
                margin = INFINITY;
            } else {
                /* p' of the processed, constrained target ([spec-notes] 8.2) */
                const float x_d = xbuf[(size_t)j * V + d];
                const float t_d = x_d >= st[j].tau ? spec_verify_ref_exp(x_d - st[j].m) : 0.0f;
                const float p_d = t_d / st[j].Sk_f;
                const float q_d = draft_probs ? draft_probs[(size_t)(q0 + j) * V + d] : 1.0f;
                const float u = u_override
                                    ? u_override[q0 + j]
                                    : spec_verify_ref_uniform(seed, 0u, (uint32_t)j, ireq,
                                                              REF_TAG_ACCEPT, 0);
                /* [spec-notes] answer code: draft_prob > 0 and target_prob / draft_prob >= uniform */
                acc = q_d > 0.0f && p_d / q_d >= u;
                margin = q_d > 0.0f ? fabs((double)u - (double)t_d / st[j].Sk / (double)q_d)
                                    : INFINITY;
            }
            if (accept_margin) accept_margin[q0 + j] = margin;
            if (!acc) {
                jstar = j;
                break;
            }
        }

        int32_t token;
        int kind = REF_RACE_NONE;
        double gap = INFINITY;
        if (greedy) {
            /* [spec-notes] 8.3 greedy: output the target argmax at the mismatch; the bonus is
             * the argmax of the bonus row. */
            token = st[jstar].amax;
        } else if (synthetic) {
            /* synthetic mode has no draft distribution: the token at j* is the target's own
             * draw from p ([MTP-eagle]: the target token is written whether accepted or not) */
            race_t r = race_row(xbuf + (size_t)jstar * V, V, st[jstar].m, st[jstar].tau,
                                st[jstar].Sk_f, NULL, -1, seed, (uint32_t)jstar, ireq, fp64);
            token = r.idx;
            gap = r.gap;
            kind = REF_RACE_TARGET;
        } else if (jstar == K) {
            /* [spec-notes] bonus token: sampled from p at the position after the last draft;
             * K = 0 is the plain Gumbel-max sample of a non-speculative request. */
            race_t r = race_row(xbuf + (size_t)K * V, V, st[K].m, st[K].tau, st[K].Sk_f, NULL, -1,
                                seed, (uint32_t)K, ireq, fp64);
            token = r.idx;
            gap = r.gap;
            kind = REF_RACE_BONUS;
        } else if (draft_probs) {
            const float *q = draft_probs + (size_t)(q0 + jstar) * V;
            race_t r = race_row(xbuf + (size_t)jstar * V, V, st[jstar].m, st[jstar].tau,
                                st[jstar].Sk_f, q, -1, seed, (uint32_t)jstar, ireq, fp64);
            kind = REF_RACE_RESIDUAL;
            if (r.idx < 0) {
                /* nothing left of max(0, p - q) after rounding: sample from p itself so that
                 * the emitted token is still a target-side draw */
                r = race_row(xbuf + (size_t)jstar * V, V, st[jstar].m, st[jstar].tau,
                             st[jstar].Sk_f, NULL, -1, seed, (uint32_t)jstar, ireq, fp64);
                kind = REF_RACE_FALLBACK;
            }
            token = r.idx;
            gap = r.gap;
        } else {
            /* [spec-notes] NO_DRAFT_PROBS: q is a point mass on d, so the residual is p with d
             * removed; an out-of-range d removes nothing. */
            const int32_t d = draft_ids[q0 + jstar];
            race_t r = race_row(xbuf + (size_t)jstar * V, V, st[jstar].m, st[jstar].tau,
                                st[jstar].Sk_f, NULL, d, seed, (uint32_t)jstar, ireq, fp64);
            if (r.idx < 0) /* V == 1 and d == 0: nothing else to draw */
                r = race_row(xbuf + (size_t)jstar * V, V, st[jstar].m, st[jstar].tau,
                             st[jstar].Sk_f, NULL, -1, seed, (uint32_t)jstar, ireq, fp64);
            token = r.idx;
            gap = r.gap;
            kind = REF_RACE_EXCLUDE;
        }

        /* [MTP-eagle] sampled[num_reqs, num_spec_steps + 1], num_sampled; [spec-notes] 9.2
         * num_rejected = num_draft - num_accepted */
        int32_t *out = sampled + (size_t)i * stride;
        for (int j = 0; j < jstar; ++j) out[j] = draft_ids[q0 + j];
        out[jstar] = token;
        for (int s = jstar + 1; s < stride; ++s) out[s] = -1;
        num_sampled[i] = jstar + 1;
        num_rejected[i] = K - jstar;
        if (race_gap) race_gap[i] = gap;
        if (race_kind) race_kind[i] = kind;
        if (jstar_out) jstar_out[i] = jstar;
        free(ybuf);
        free(xbuf);
    }
    return REF_OK;
}

/*
 * Draft distributions from draft logits ([spec-in-vllm] 7.1 probabilistic draft sampling keeps
 * the draft logits; 7.4 block stats over target and draft logits): for draft row qrow of request
 * i, q = softmax(draft_logits / T_i), with the request's own temperature (1 for a greedy request,
 * whose q is never used):
 *   x'_v = fl(dl_v * (1 / T_i)), m_d = max_v x'_v, S_d = (float) sum_v (double) exp(x'_v - m_d),
 *   q_v = fl(exp(x'_v - m_d) / S_d),
 * the same binary32 steps as the target's p = t / S. Rows of an inconsistent batch are skipped.
 * q_out: [num_draft_tokens, V].
 */
void spec_verify_ref_draft_probs(const void *draft_logits, int logits_bf16, int vocab_size,
                                 const int32_t *cu_num_draft, const float *temperature,
                                 const uint8_t *is_greedy, int num_reqs, float *q_out)
{
    const int V = vocab_size;
    for (int i = 0; i < num_reqs; ++i) {
        const float T = temperature[i];
        const int greedy = is_greedy[i] != 0 || !(T > 0.0f);
        const float invT = greedy ? 1.0f : 1.0f / T;
        for (int32_t r = cu_num_draft[i]; r < cu_num_draft[i + 1]; ++r) {
            const size_t base = (size_t)r * V;
            float m = -INFINITY;
            for (int v = 0; v < V; ++v) {
                float x = logit_at(draft_logits, logits_bf16, base + (size_t)v) * invT;
                if (x > m) m = x;
            }
            double S = 0.0;
            for (int v = 0; v < V; ++v) {
                float x = logit_at(draft_logits, logits_bf16, base + (size_t)v) * invT;
                S += (double)spec_verify_ref_exp(x - m);
            }
            const float S_f = (float)S;
            for (int v = 0; v < V; ++v) {
                float x = logit_at(draft_logits, logits_bf16, base + (size_t)v) * invT;
                q_out[base + (size_t)v] = spec_verify_ref_exp(x - m) / S_f;
            }
        }
    }
}

/* Residual weights of one row as the race uses them (for identity checks):
 * t_v = exp(x_v - m), rr_v = fma(-S, q_v, t_v); also returns m and S (binary32). */
void spec_verify_ref_residual_row(const void *logits_row, int logits_bf16, int vocab_size,
                                  float invT, const float *q, float *t_out, float *rr_out,
                                  float *m_out, float *S_out)
{
    float *y = (float *)malloc((size_t)vocab_size * sizeof(float));
    float *x = (float *)malloc((size_t)vocab_size * sizeof(float));
    processed_row(logits_row, logits_bf16, 0, vocab_size, invT, 0.0f, NULL, NULL, 0, y, x);
    row_stats_t st = row_stats(y, x, vocab_size);
    for (int v = 0; v < vocab_size; ++v) {
        t_out[v] = spec_verify_ref_exp(x[v] - st.m);
        if (rr_out) rr_out[v] = fmaf(-st.S_f, q[v], t_out[v]);
    }
    *m_out = st.m;
    *S_out = st.S_f;
    free(y);
    free(x);
}

/* The sampling constraints of one processed row x[0..V) (for the checks of select_row):
 * writes the threshold tau (kept: x >= tau), the kept mass Sk (double) and the top-p margin. */
void spec_verify_ref_select_row(const float *x, int V, int top_k, float top_p, float *tau,
                                double *Sk, double *margin)
{
    row_stats_t st = row_stats(x, x, V);
    select_row(x, V, top_k, top_p, &st);
    *tau = st.tau;
    *Sk = st.Sk;
    *margin = st.margin;
}

/* Element-wise exp / log over arrays (for the accuracy checks of the two functions). */
void spec_verify_ref_exp_n(const float *in, float *out, int64_t n)
{
    for (int64_t k = 0; k < n; ++k) out[k] = spec_verify_ref_exp(in[k]);
}

void spec_verify_ref_log_n(const float *in, float *out, int64_t n)
{
    for (int64_t k = 0; k < n; ++k) out[k] = spec_verify_ref_log(in[k]);
}

/* Race clocks of tokens v in [0, n) of (request ireq, position j). */
void spec_verify_ref_race_clocks(uint64_t seed, uint32_t j, uint32_t ireq, int32_t n, float *out)
{
    for (int32_t v = 0; v < n; ++v) out[v] = spec_verify_ref_race_clock(seed, j, ireq, v);
}

/* The same in binary64. */
void spec_verify_ref_race_clocks64(uint64_t seed, uint32_t j, uint32_t ireq, int32_t n, double *out)
{
    for (int32_t v = 0; v < n; ++v) out[v] = spec_verify_ref_race_clock64(seed, j, ireq, v);
}

/* binary64 log over an array (for the accuracy checks). */
void spec_verify_ref_log64_n(const double *in, double *out, int64_t n)
{
    for (int64_t k = 0; k < n; ++k) out[k] = spec_verify_ref_log64(in[k]);
}

/* ------------------------------------------------------------------------------------ */
/* Vocabulary-sharded verification. The logits (and draft probabilities) of every row are   */
/* split by vocabulary over `world` ranks, rank r holding the columns [v0_r, v0_r + Vs_r)   */
/* with v0_r a multiple of 64 (race-clock groups stay whole). Two exchanges reproduce the   */
/* unsharded step: the shard statistics of every row (after which every rank evaluates the  */
/* same acceptance tests), then each shard's best race key at the row of the first          */
/* rejection; the largest key over the shards is the winner of the whole row's race.        */
/* Plain processing only (x = logit / T).                                                   */
/* ------------------------------------------------------------------------------------ */
typedef struct {
    float ymax;   /* largest logit of the shard */
    int32_t amax; /* its first global index */
    double s;     /* sum over the shard of exp(x_v - fl(ymax / T)), double, index order */
    float ld;     /* logit of the row's draft token if the shard holds it, else NaN */
    float qd;     /* its draft probability (1 without draft probabilities), else NaN */
} ref_shard_stats_t;

typedef struct {
    int32_t jstar;   /* first rejection (K if none): the same on every rank */
    int32_t token;   /* a greedy request's token (the combined argmax), else -1 */
    float res_key;   /* the shard's best residual / exclusion key, */
    int32_t res_idx; /* and its global index (-1: no candidate in the shard) */
    float p_key;     /* the shard's best key of the race over p (the fallback and the bonus) */
    int32_t p_idx;
} ref_shard_race_t;

void spec_verify_ref_shard_stats(const void *logits, int logits_bf16, int shard_vocab, int v0,
                                 const int32_t *draft_ids, const float *draft_probs,
                                 const int32_t *cu_num_draft, const float *temperature,
                                 const uint8_t *is_greedy, int num_reqs,
                                 ref_shard_stats_t *out)
{
    const int Vs = shard_vocab;
    for (int i = 0; i < num_reqs; ++i) {
        const int q0 = cu_num_draft[i], K = cu_num_draft[i + 1] - q0;
        const float T = temperature[i];
        const int greedy = is_greedy[i] != 0 || !(T > 0.0f);
        const float invT = greedy ? 1.0f : 1.0f / T;
        for (int j = 0; j <= K; ++j) {
            const size_t row = (size_t)q0 + (size_t)i + (size_t)j, base = row * (size_t)Vs;
            ref_shard_stats_t st;
            st.ymax = -INFINITY;
            st.amax = v0;
            for (int v = 0; v < Vs; ++v) {
                const float l = logit_at(logits, logits_bf16, base + (size_t)v);
                if (l > st.ymax) {
                    st.ymax = l;
                    st.amax = v0 + v;
                }
            }
            const float mr = st.ymax * invT;
            st.s = 0.0;
            for (int v = 0; v < Vs; ++v)
                st.s += (double)spec_verify_ref_exp(logit_at(logits, logits_bf16, base + (size_t)v) * invT - mr);
            st.ld = NAN;
            st.qd = NAN;
            if (j < K) {
                const int32_t d = draft_ids[q0 + j];
                if (d >= v0 && d < v0 + Vs) {
                    st.ld = logit_at(logits, logits_bf16, base + (size_t)(d - v0));
                    st.qd = draft_probs ? draft_probs[(size_t)(q0 + j) * Vs + (size_t)(d - v0)] : 1.0f;
                }
            }
            out[row] = st;
        }
    }
}

/* The best key of the shard's race at row `row` (global indices; lowest index on equal keys). */
static void shard_race_best(const void *logits, int bf16, int Vs, int v0, size_t row, float invT,
                            float m, float S_f, const float *q, int32_t exclude, uint64_t seed,
                            uint32_t j, uint32_t ireq, float *key, int32_t *idx)
{
    *key = -INFINITY;
    *idx = -1;
    for (int v = 0; v < Vs; ++v) {
        const int32_t g = v0 + v;
        if (g == exclude) continue;
        const float x = logit_at(logits, bf16, row * (size_t)Vs + (size_t)v) * invT;
        const float t = spec_verify_ref_exp(x - m);
        float w = t;
        if (q) {
            w = fmaf(-S_f, q[v], t);
            if (!(w > 0.0f)) continue;
        }
        const float k = w / spec_verify_ref_race_clock(seed, j, ireq, g);
        if (*idx < 0 || k > *key) {
            *key = k;
            *idx = g;
        }
    }
}

void spec_verify_ref_shard_race(const void *logits, int logits_bf16, int shard_vocab, int v0,
                                int vocab_size, const ref_shard_stats_t *all_stats, int world,
                                const int32_t *draft_ids, const float *draft_probs,
                                const int32_t *cu_num_draft, const float *temperature,
                                const uint8_t *is_greedy, uint64_t seed, uint32_t req_index_base,
                                int num_reqs, int num_draft_tokens, ref_shard_race_t *out)
{
    const int Vs = shard_vocab, V = vocab_size;
    const size_t R = (size_t)num_draft_tokens + (size_t)num_reqs;
    for (int i = 0; i < num_reqs; ++i) {
        const int q0 = cu_num_draft[i], K = cu_num_draft[i + 1] - q0;
        const uint32_t ireq = req_index_base + (uint32_t)i;
        const float T = temperature[i];
        const int greedy = is_greedy[i] != 0 || !(T > 0.0f);
        const float invT = greedy ? 1.0f : 1.0f / T;
        float m[K + 1], S_f[K + 1];
        int32_t amax[K + 1];
        int jstar = K;
        for (int j = 0; j <= K; ++j) {
            const size_t row = (size_t)q0 + (size_t)i + (size_t)j;
            /* combine the shards: the largest logit (first index on ties) and the sum */
            float ymax = -INFINITY;
            amax[j] = 0;
            for (int r = 0; r < world; ++r) {
                const ref_shard_stats_t *st = all_stats + (size_t)r * R + row;
                if (st->ymax > ymax || (st->ymax == ymax && st->amax < amax[j])) {
                    ymax = st->ymax;
                    amax[j] = st->amax;
                }
            }
            m[j] = ymax * invT;
            double S = 0.0;
            for (int r = 0; r < world; ++r) {
                const ref_shard_stats_t *st = all_stats + (size_t)r * R + row;
                S += st->s * exp((double)(st->ymax * invT) - (double)m[j]);
            }
            S_f[j] = (float)S;
            if (j < K && jstar == K) {
                const int32_t d = draft_ids[q0 + j];
                int acc;
                if (greedy) {
                    acc = d == amax[j];
                } else if (d < 0 || d >= V) {
                    acc = 0;
                } else {
                    float ld = NAN, qd = NAN;
                    for (int r = 0; r < world; ++r) {
                        const ref_shard_stats_t *st = all_stats + (size_t)r * R + row;
                        if (st->ld == st->ld) {
                            ld = st->ld;
                            qd = st->qd;
                        }
                    }
                    const float t_d = spec_verify_ref_exp(ld * invT - m[j]);
                    const float u = spec_verify_ref_uniform(seed, 0u, (uint32_t)j, ireq, REF_TAG_ACCEPT, 0);
                    acc = qd > 0.0f && (t_d / S_f[j]) / qd >= u;
                }
                if (!acc) jstar = j;
            }
        }
        ref_shard_race_t o;
        o.jstar = jstar;
        o.token = greedy ? amax[jstar] : -1;
        o.res_key = o.p_key = -INFINITY;
        o.res_idx = o.p_idx = -1;
        if (!greedy) {
            const size_t row = (size_t)q0 + (size_t)i + (size_t)jstar;
            if (jstar < K) {
                const float *q = draft_probs ? draft_probs + (size_t)(q0 + jstar) * Vs : NULL;
                const int32_t excl = draft_probs ? -1 : draft_ids[q0 + jstar];
                shard_race_best(logits, logits_bf16, Vs, v0, row, invT, m[jstar], S_f[jstar], q, excl,
                                seed, (uint32_t)jstar, ireq, &o.res_key, &o.res_idx);
            }
            shard_race_best(logits, logits_bf16, Vs, v0, row, invT, m[jstar], S_f[jstar], NULL, -1,
                            seed, (uint32_t)jstar, ireq, &o.p_key, &o.p_idx);
        }
        out[i] = o;
    }
}

/* The winner over the shards, and the emitted row: the residual (or exclusion) race when j* < K
 * and some shard has a candidate, else the race over p. */
void spec_verify_ref_shard_finish(const ref_shard_race_t *all_races, int world,
                                  const int32_t *draft_ids, const int32_t *cu_num_draft,
                                  int num_reqs, int max_spec_len, int32_t *sampled,
                                  int32_t *num_sampled, int32_t *num_rejected)
{
    const int stride = max_spec_len + 1;
    for (int i = 0; i < num_reqs; ++i) {
        const int q0 = cu_num_draft[i], K = cu_num_draft[i + 1] - q0;
        const ref_shard_race_t *o0 = all_races + i;
        const int jstar = o0->jstar;
        int32_t token = o0->token;
        if (token < 0) {
            float best = -INFINITY;
            int32_t bi = -1;
            if (jstar < K)
                for (int r = 0; r < world; ++r) {
                    const ref_shard_race_t *o = all_races + (size_t)r * num_reqs + i;
                    if (o->res_idx >= 0 && (bi < 0 || o->res_key > best || (o->res_key == best && o->res_idx < bi))) {
                        best = o->res_key;
                        bi = o->res_idx;
                    }
                }
            if (bi < 0)
                for (int r = 0; r < world; ++r) {
                    const ref_shard_race_t *o = all_races + (size_t)r * num_reqs + i;
                    if (o->p_idx >= 0 && (bi < 0 || o->p_key > best || (o->p_key == best && o->p_idx < bi))) {
                        best = o->p_key;
                        bi = o->p_idx;
                    }
                }
            token = bi;
        }
        int32_t *out = sampled + (size_t)i * stride;
        for (int j = 0; j < jstar; ++j) out[j] = draft_ids[q0 + j];
        out[jstar] = token;
        for (int s = jstar + 1; s < stride; ++s) out[s] = -1;
        num_sampled[i] = jstar + 1;
        num_rejected[i] = K - jstar;
    }
}
