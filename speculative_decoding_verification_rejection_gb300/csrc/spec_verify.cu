// GB300 (sm_103a) implementation of the speculative-decoding verification sampler behind the
// C ABI declared in include/spec_verify.h.
//
// One call = four kernels on the caller's stream, no allocation, no host synchronisation:
//   1. plan  (1 CTA)    validate cu_num_draft, map every logit row to (request, j), list the
//                       sampling (non-greedy) requests, clear the cross-CTA counters.
//   2. stats (4 waves)  stream every logit once, the flattened [rows x V] array split evenly
//                       over the CTAs, one partial (max, sum of exp, argmax) per row segment
//                       ([spec-in-vllm] 7.4 block stats).
//   3. finalize (warp per row) combine a row's partials: m = max x, S = sum exp(x - m), raw
//                       argmax; run the row's acceptance test ([spec-notes] 8.3 and the
//                       NO_DRAFT_PROBS answer code); the warp that completes a request's last row
//                       finds the first rejection j* ([MTP-eagle] _rejection_sample_kernel),
//                       emits greedy requests outright and records for sampling requests which
//                       row to race.
//   4. race  (2 waves)  the raced rows -- one per sampling request -- concatenated and split
//                       evenly over the CTAs: the exponential race over the residual
//                       max(0, p - q), over p without the rejected draft, or over p for the bonus
//                       / non-speculative draw ([spec-notes] residual and NO_DRAFT_PROBS answers,
//                       [spec-in-vllm] 7.3); the CTA that completes a request's race emits
//                       sampled / num_sampled / num_rejected.
// Only the emitted row of a request is raced: a residual that is never emitted cannot change
// any output, so its logits and q row are never read twice.
#include <cuda_runtime.h>

#include <algorithm>
#include <climits>
#include <cstddef>
#include <cstdint>
#include <mutex>
#include <new>
#include <vector>

#include "spec_verify.h"
#include "sv_device.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kPlanThreads = 1024;
constexpr int kMinChunk = 2048;     // smallest elements per CTA (bounds the partial buffers)
constexpr int kStatsWaves = 4;      // automatic statistics grid: this many full waves of CTAs
constexpr int kRaceWaves = 2;       // automatic race grid
constexpr int kFixedChunk = 16384;  // chunk of the static-scratch entry point (both kernels)
constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kInf = __builtin_huge_valf();

enum : int32_t { kFlagGreedy = 1, kFlagBonus = 2, kFlagKShift = 8 };  // flags = g | b | K << 8

struct __align__(16) RowInfo {
    int32_t req;    // request index within the call
    int32_t j;      // position, K = bonus
    int32_t flags;  // kFlagGreedy | kFlagBonus | K << kFlagKShift
    float invT;     // 1 / T (1 for greedy rows)
};

struct __align__(16) RowStat {
    float m;          // max_v x_v
    float S;          // sum_v exp(x_v - m)
    int32_t amax;     // raw-logit argmax, lowest index
    int32_t acc;      // acceptance of the row's draft (bonus rows: 1)
    uint32_t seed_p;  // race key of the argmax token in a race over p (encoded), for screening
    uint32_t seed_r;  // its key in the residual race (encoded; none on bonus rows or if rr <= 0)
    uint32_t pad[2];
};

struct __align__(16) ReqState {  // what the race of a sampling request needs
    int32_t jstar;   // first rejected position (K if every draft was accepted)
    int32_t K;
    int32_t q0;      // cu_num_draft[i]
    int32_t row;     // the raced logit row
    float m, S, invT;
    uint32_t seed;   // screening seed of the race (encoded key)
    uint32_t seed_p; // seed of a race over p on the same row (the empty-residual fallback)
    int32_t excl;    // token removed from the race (the rejected draft without q), else -1
    int32_t pad[2];
};

struct __align__(16) StatPart {
    float L;       // max raw logit of the segment
    float s;       // sum of 2^((l - L) c) over the segment
    int32_t idx;   // lowest index of L
    int32_t pad;
};

struct __align__(8) RacePart {
    float key;
    int32_t idx;   // -1: no candidate
};

// ---------------------------------------------------------------------------------------
// element loads
// ---------------------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float at(const float *p, size_t k) { return __ldg(p + k); }
};
template <> struct Elem<uint16_t> {
    static __device__ __forceinline__ float at(const uint16_t *p, size_t k)
    {
        return __uint_as_float(static_cast<uint32_t>(__ldg(p + k)) << 16);
    }
};

__device__ __forceinline__ uint4 ldg_v4(const void *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// ---------------------------------------------------------------------------------------
// race keys
// ---------------------------------------------------------------------------------------
// Keys as order-preserving unsigned integers, so that atomicMax can share a threshold.
__device__ __forceinline__ unsigned key_enc(float f)
{
    const unsigned b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_dec(unsigned e)
{
    return __uint_as_float((e & 0x80000000u) ? (e & 0x7FFFFFFFu) : ~e);
}
constexpr unsigned kKeyNone = 0x007FFFFFu;  // key_enc(-inf): no threshold yet

// Full key of a token (the definition, bit for bit): over p, x - log E; over the residual,
// log(fma(-S, q, exp(x - m))) - log E; E the token's race clock. Returns false if the token is
// not a candidate (residual weight <= 0).
template <bool kResidual>
__device__ __forceinline__ bool race_key(float x, float qv, float E, float m, float S, float &key)
{
    if constexpr (kResidual) {
        const float t = sv::exp_f32(__fsub_rn(x, m));
        const float rr = __fmaf_rn(-S, qv, t);
        if (!(rr > 0.0f)) return false;
        key = __fsub_rn(sv::log_f32(rr), sv::log_f32(E));
    } else {
        key = __fsub_rn(x, sv::log_f32(E));
    }
    return true;
}

__device__ __forceinline__ uint32_t pick_word(const sv::Philox4 &r, int k)
{
    return (k & 2) ? ((k & 1) ? r.w : r.z) : ((k & 1) ? r.y : r.x);
}

// Race clock of slot s of a block from its head words (W word, slot a) and the slot call's word
// (unused for s == a): E_min = -log(W) / 16, plus -log(U_s) for s != a.
__device__ __forceinline__ float race_clock(uint32_t w_head, int a, int s, uint32_t w_slot)
{
    const float emin = __fmul_rn(-sv::log_f32(sv::uniform_from_word(w_head)), 0.0625f);
    if (s == a) return emin;
    return __fadd_rn(emin, -sv::log_f32(sv::uniform_from_word(w_slot)));
}

// Clock of token v at position j of request ireq (two Philox calls; used off the hot path).
__device__ __forceinline__ float token_clock(int v, uint32_t j, uint32_t ireq, uint64_t seed)
{
    const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    const uint32_t g = static_cast<uint32_t>(v) >> 4;
    const int s = v & 15;
    const sv::Philox4 h = sv::philox4x32_10(g, j, ireq, sv::kClockHead, k0, k1);
    const int a = static_cast<int>(h.y & 15u);
    uint32_t w = 0u;
    if (s != a) w = pick_word(sv::philox4x32_10(g, j, ireq, sv::kClockHead + 1u + (s >> 2), k0, k1), s & 3);
    return race_clock(h.x, a, s, w);
}

__device__ __forceinline__ void emit_row(int i, int jstar, int K, int q0, int token,
                                         const int32_t *__restrict__ draft_ids,
                                         int32_t *__restrict__ sampled, int stride,
                                         int32_t *__restrict__ num_sampled,
                                         int32_t *__restrict__ num_rejected, int tid, int nthreads)
{
    int32_t *out = sampled + static_cast<size_t>(i) * stride;
    for (int s = tid; s < stride; s += nthreads)
        out[s] = s < jstar ? draft_ids[q0 + s] : (s == jstar ? token : -1);
    if (tid == 0) {
        num_sampled[i] = jstar + 1;
        num_rejected[i] = jstar < 0 ? 0 : K - jstar;
    }
}

// ---------------------------------------------------------------------------------------
// 1. plan
// ---------------------------------------------------------------------------------------
// Scratch words per request: rows-done counter, race counter, race threshold, sampling list.
struct ReqWords {
    unsigned *rows_done, *race_counter, *race_thr;
    int *rand_req, *n_rand;
};

__global__ void __launch_bounds__(kPlanThreads)
sv_plan_kernel(const int32_t *__restrict__ cu, const float *__restrict__ temperature,
               const uint8_t *__restrict__ is_greedy, int num_reqs, int num_draft_tokens,
               int kmax, RowInfo *__restrict__ rowinfo, ReqWords rw,
               int32_t *__restrict__ sampled, int stride,
               int32_t *__restrict__ num_sampled, int32_t *__restrict__ num_rejected,
               unsigned *__restrict__ flags)
{
    __shared__ int bad;
    __shared__ int warp_count[kPlanThreads / 32];
    __shared__ int s_base;
    if (threadIdx.x == 0) {
        bad = (cu[0] != 0) || (cu[num_reqs] != num_draft_tokens);
        s_base = 0;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int i0 = 0; i0 < num_reqs; i0 += blockDim.x) {
        const int i = i0 + threadIdx.x;
        bool sampling = false;
        if (i < num_reqs) {
            rw.rows_done[i] = 0u;
            rw.race_counter[i] = 0u;
            rw.race_thr[i] = kKeyNone;
            const int lo = cu[i], hi = cu[i + 1];
            const int K = hi - lo;
            if (K < 0 || K > kmax || lo < 0 || hi > num_draft_tokens) {
                bad = 1;
            } else {
                const float T = temperature[i];
                const bool greedy = is_greedy[i] != 0 || !(T > 0.0f);
                const float invT = greedy ? 1.0f : __frcp_rn(T);
                const int32_t f = (greedy ? kFlagGreedy : 0) | (K << kFlagKShift);
                for (int j = 0; j <= K; ++j)
                    rowinfo[lo + i + j] = RowInfo{i, j, f | (j == K ? kFlagBonus : 0), invT};
                sampling = !greedy;
            }
        }
        // list the sampling requests in index order (ballot within warps, scan across warps)
        const unsigned m = __ballot_sync(0xFFFFFFFFu, sampling);
        if (lane == 0) warp_count[warp] = __popc(m);
        __syncthreads();
        if (warp == 0) {
            const int c = warp_count[lane];
            int x = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
                if (lane >= o) x += y;
            }
            warp_count[lane] = x - c;  // exclusive prefix
        }
        __syncthreads();
        if (sampling)
            rw.rand_req[s_base + warp_count[warp] + __popc(m & ((1u << lane) - 1u))] = i;
        __syncthreads();
        if (threadIdx.x == blockDim.x - 1)
            s_base += warp_count[warp] + __popc(m);
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        *rw.n_rand = bad ? 0 : s_base;
        flags[0] = bad ? 1u : 0u;
        if (bad) atomicOr(&flags[1], SV_ERR_BATCH);
    }
    if (bad)  // an inconsistent batch emits nothing for any request
        for (int i = threadIdx.x; i < num_reqs; i += blockDim.x)
            emit_row(i, -1, 0, 0, -1, nullptr, sampled, stride, num_sampled, num_rejected, 0, 1);
}

// ---------------------------------------------------------------------------------------
// 2. row statistics, acceptance test, request completion
// ---------------------------------------------------------------------------------------
struct OnlineMax {
    float L = -kInf;   // running max of raw logits
    float s = 0.0f;    // running sum of 2^((l - L) c)
    float Lc = 0.0f;   // L * c once L is finite (0 before, so that -inf logits add 2^-inf = 0)
    int best_e = -1;   // element where L was first reached (scalar path), or -1
    int best_u = -1;   // first vector of the batch where L was first reached, or -1
};

// Fold one logit at index e (head / tail of a misaligned segment; indices increase).
__device__ __forceinline__ void fold1(OnlineMax &st, float l, int e, float c)
{
    if (l > st.L) {
        st.s = st.s == 0.0f ? 0.0f : st.s * sv::ex2_approx((st.L - l) * c);
        st.L = l;
        st.Lc = l * c;
        st.best_e = e;
        st.best_u = -1;
    }
    st.s += sv::ex2_approx(fmaf(l, c, -st.Lc));
}

template <typename T>
__device__ __forceinline__ void unpack(const uint4 &w, float (&l)[16 / sizeof(T)])
{
    if constexpr (sizeof(T) == 2) {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            l[2 * h] = __uint_as_float(ws[h] << 16);
            l[2 * h + 1] = __uint_as_float(ws[h] & 0xFFFF0000u);
        }
    } else {
        l[0] = __uint_as_float(w.x);
        l[1] = __uint_as_float(w.y);
        l[2] = __uint_as_float(w.z);
        l[3] = __uint_as_float(w.w);
    }
}

// Fold a batch of NV 16-byte vectors (vectors u0, u0 + kThreads, ...; element indices increase
// with the vector) without branches: the batch max first, then one rescale of the running sum,
// then the sum of 2^((l - L) c). Only the batch that first reached the max is recorded; its
// lowest index is recovered at the end of the segment.
template <typename T, int NV>
__device__ __forceinline__ void fold_batch(OnlineMax &st, const uint4 (&w)[NV], int nv, int u0,
                                           float c)
{
    constexpr int kVec = 16 / sizeof(T);
    float mx = -kInf;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        if (k < nv) {
            float l[kVec];
            unpack<T>(w[k], l);
#pragma unroll
            for (int h = 0; h < kVec; ++h) mx = fmaxf(mx, l[h]);
        }
    }
    const bool up = mx > st.L;
    st.s *= sv::ex2_approx(up ? (st.L - mx) * c : 0.0f);  // L = -inf: 2^-inf = 0 (s was 0)
    st.best_u = up ? u0 : st.best_u;
    st.best_e = up ? -1 : st.best_e;
    st.L = up ? mx : st.L;
    st.Lc = st.L > -kInf ? st.L * c : 0.0f;
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int k = 0; k < NV; ++k) {
        if (k < nv) {
            float l[kVec];
            unpack<T>(w[k], l);
#pragma unroll
            for (int h = 0; h < kVec; ++h)
                ((h & 1) ? s1 : s0) += sv::ex2_approx(fmaf(l[h], c, -st.Lc));
        }
    }
    st.s += s0 + s1;
}

__device__ __forceinline__ void combine_stat(float &L, float &s, int &idx, float L2, float s2,
                                             int i2, float c)
{
    const float Lm = fmaxf(L, L2);
    const float a = s == 0.0f ? 0.0f : s * sv::ex2_approx((L - Lm) * c);
    const float b = s2 == 0.0f ? 0.0f : s2 * sv::ex2_approx((L2 - Lm) * c);
    const int id = L > L2 ? idx : (L2 > L ? i2 : min(idx, i2));
    L = Lm;
    s = a + b;
    idx = id;
}

// Warp then block reduction of (L, s, idx); result valid in thread 0.
__device__ __forceinline__ void block_reduce_stat(float &L, float &s, int &idx, float c)
{
    __shared__ float sh_L[kThreads / 32], sh_s[kThreads / 32];
    __shared__ int sh_i[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float L2 = __shfl_xor_sync(0xFFFFFFFFu, L, o);
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, idx, o);
        combine_stat(L, s, idx, L2, s2, i2, c);
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // sh_* may still be read by the previous segment's reduction
    if (lane == 0) {
        sh_L[warp] = L;
        sh_s[warp] = s;
        sh_i[warp] = idx;
    }
    __syncthreads();
    if (warp == 0) {
        L = lane < kThreads / 32 ? sh_L[lane] : -kInf;
        s = lane < kThreads / 32 ? sh_s[lane] : 0.0f;
        idx = lane < kThreads / 32 ? sh_i[lane] : INT_MAX;
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {
            const float L2 = __shfl_xor_sync(0xFFFFFFFFu, L, o);
            const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
            const int i2 = __shfl_xor_sync(0xFFFFFFFFu, idx, o);
            combine_stat(L, s, idx, L2, s2, i2, c);
        }
    }
}

// Acceptance test of the row's draft ([spec-notes] answer code: draft_prob > 0 and
// target_prob / draft_prob >= uniform; greedy: d == argmax, [spec-notes] 8.3). One thread.
template <typename T>
__device__ __forceinline__ int accept_test(const T *rp, int V, const RowInfo &ri, int row, float m,
                                           float S, int amax, const int32_t *__restrict__ draft_ids,
                                           const float *__restrict__ q, uint64_t seed,
                                           uint32_t req_base)
{
    if (ri.flags & kFlagBonus) return 1;
    const int qrow = row - ri.req;  // cu_num_draft[i] + j
    const int d = draft_ids[qrow];
    if (ri.flags & kFlagGreedy) return d == amax;
    if (d < 0 || d >= V) return 0;
    const float x_d = __fmul_rn(Elem<T>::at(rp, d), ri.invT);
    const float t_d = sv::exp_f32(__fsub_rn(x_d, m));
    const float p_d = __fdiv_rn(t_d, S);
    const float q_d = q ? __ldg(q + static_cast<size_t>(qrow) * V + d) : 1.0f;
    const sv::Philox4 r = sv::philox4x32_10(0u, static_cast<uint32_t>(ri.j),
                                            req_base + static_cast<uint32_t>(ri.req),
                                            sv::kTagAccept, static_cast<uint32_t>(seed),
                                            static_cast<uint32_t>(seed >> 32));
    const float u = sv::uniform_from_word(r.x);
    return (q_d > 0.0f) && (__fdiv_rn(p_d, q_d) >= u);
}

struct StatsOut {  // what the statistics kernel writes besides per-row partials
    RowStat *rowstat;
    ReqState *reqstate;
    unsigned *rows_done;
    int32_t *sampled, *num_sampled, *num_rejected;
    int stride;
    float *opt_max, *opt_sum;
    int32_t *opt_amax;
};

// The request's last row has been finalised (one thread): find j*, emit a greedy request, or
// record the race of a sampling request.
__device__ __noinline__ void complete_request(int i, int row0, int K, bool greedy, float invT,
                                              const int32_t *__restrict__ draft_ids, bool has_q,
                                              const StatsOut &o)
{
    const int q0 = row0 - i;
    int js = K;
    for (int jj = 0; jj < K; ++jj)
        if (__ldcg(&o.rowstat[row0 + jj].acc) == 0) {
            js = jj;
            break;
        }
    const RowStat *rs = &o.rowstat[row0 + js];
    const int amax = __ldcg(&rs->amax);
    if (greedy) {  // [spec-notes] 8.3: the target argmax at the mismatch, or of the bonus row
        emit_row(i, js, K, q0, amax, draft_ids, o.sampled, o.stride, o.num_sampled,
                 o.num_rejected, 0, 1);
        return;
    }
    const bool residual = js < K && has_q;
    const int excl = (js < K && !has_q) ? draft_ids[q0 + js] : -1;
    const uint32_t seed_p = __ldcg(&rs->seed_p);
    const uint32_t seed = residual ? __ldcg(&rs->seed_r) : (amax == excl ? kKeyNone : seed_p);
    o.reqstate[i] = ReqState{js, K, q0, row0 + js, __ldcg(&rs->m), __ldcg(&rs->S), invT, seed,
                             seed_p, excl, {0, 0}};
}

// Finalise row `row` from its combined statistics (one thread): m, S, the argmax, the acceptance
// of the row's draft and the race's screening seeds (the argmax token's keys); the finaliser of
// a request's last row completes the request.
template <typename T>
__device__ __forceinline__ void finalize_row(const T *rp, int V, int row, const RowInfo &ri,
                                             float L, float s, int idx,
                                             const int32_t *__restrict__ draft_ids,
                                             const float *__restrict__ q, uint64_t seed,
                                             uint32_t req_base, const StatsOut &o)
{
    const float m = __fmul_rn(L, ri.invT);  // = max_v fl(l_v / T): rounding is monotone
    const int amax = idx == INT_MAX ? 0 : idx;
    const int acc = accept_test<T>(rp, V, ri, row, m, s, amax, draft_ids, q, seed, req_base);
    uint32_t seed_p = kKeyNone, seed_r = kKeyNone;
    if (!(ri.flags & kFlagGreedy)) {
        const float x = __fmul_rn(Elem<T>::at(rp, amax), ri.invT);
        const float E = token_clock(amax, static_cast<uint32_t>(ri.j),
                                    req_base + static_cast<uint32_t>(ri.req), seed);
        float key;
        if (race_key<false>(x, 0.0f, E, m, s, key)) seed_p = key_enc(key);
        if (q && !(ri.flags & kFlagBonus)) {
            const float qv = __ldg(q + static_cast<size_t>(row - ri.req) * V + amax);
            if (race_key<true>(x, qv, E, m, s, key)) seed_r = key_enc(key);
        }
    }
    o.rowstat[row] = RowStat{m, s, amax, acc, seed_p, seed_r, {0u, 0u}};
    if (o.opt_max) o.opt_max[row] = m;
    if (o.opt_sum) o.opt_sum[row] = s;
    if (o.opt_amax) o.opt_amax[row] = amax;

    const int K = ri.flags >> kFlagKShift;
    __threadfence();
    if (atomicAdd(&o.rows_done[ri.req], 1u) == static_cast<unsigned>(K)) {
        __threadfence();
        o.rows_done[ri.req] = 0u;
        complete_request(ri.req, row - ri.j, K, (ri.flags & kFlagGreedy) != 0, ri.invT, draft_ids,
                         q != nullptr, o);
    }
}

// Segment [b, e) of row `row`, by the whole CTA: stream the logits in batches of four 16-byte
// loads per thread (the row's parameters arrive while the first batch is in flight), reduce,
// and publish the segment's partial statistics.
template <typename T>
__device__ __forceinline__ void stats_segment(const T *__restrict__ logits, int V, int row, int b,
                                              int e, int seg, int maxseg,
                                              const RowInfo *__restrict__ rowinfo,
                                              StatPart *__restrict__ part)
{
    const T *rp = logits + static_cast<size_t>(row) * static_cast<size_t>(V);
    constexpr int kVec = 16 / sizeof(T);
    constexpr int kU = 4;
    const uintptr_t addr = reinterpret_cast<uintptr_t>(rp + b);
    const int head = static_cast<int>(((16u - (addr & 15u)) & 15u) / sizeof(T));
    const int a0 = min(e, b + head);
    const int nvec = (e - a0) / kVec;
    const int a1 = a0 + nvec * kVec;
    const char *vbase = reinterpret_cast<const char *>(rp + a0);

    uint4 w[kU];
    int u0 = static_cast<int>(threadIdx.x);
#pragma unroll
    for (int k = 0; k < kU; ++k) {
        const int u = u0 + k * kThreads;
        w[k] = u < nvec ? ldg_v4(vbase + static_cast<size_t>(u) * 16) : make_uint4(0, 0, 0, 0);
    }
    const RowInfo ri = rowinfo[row];
    const float c = ri.invT * kLog2e;

    OnlineMax st;
    for (int ee = b + threadIdx.x; ee < a0; ee += kThreads) fold1(st, Elem<T>::at(rp, ee), ee, c);
    while (u0 < nvec) {
        const int nv = min(kU, (nvec - u0 + kThreads - 1) / kThreads);
        fold_batch<T, kU>(st, w, nv, u0, c);
        u0 += kThreads * kU;
#pragma unroll
        for (int k = 0; k < kU; ++k) {
            const int u = u0 + k * kThreads;
            w[k] = u < nvec ? ldg_v4(vbase + static_cast<size_t>(u) * 16) : make_uint4(0, 0, 0, 0);
        }
    }
    for (int ee = a1 + threadIdx.x; ee < e; ee += kThreads) fold1(st, Elem<T>::at(rp, ee), ee, c);

    // lowest index where this thread's max occurs
    int idx = st.best_e >= 0 ? st.best_e : INT_MAX;
    if (st.best_u >= 0) {
        for (int k = 0; k < kU && idx == INT_MAX; ++k) {
            const int u = st.best_u + k * kThreads;
            if (u >= nvec) break;
            float l[kVec];
            unpack<T>(ldg_v4(vbase + static_cast<size_t>(u) * 16), l);
#pragma unroll
            for (int h = kVec - 1; h >= 0; --h)
                if (l[h] == st.L) idx = a0 + u * kVec + h;
        }
    }
    float L = st.L, s = st.s;
    block_reduce_stat(L, s, idx, c);
    if (threadIdx.x == 0) part[static_cast<size_t>(row) * maxseg + seg] = StatPart{L, s, idx, 0};
}

// Row statistics over the flattened [rows x V] logits, split evenly: CTA k streams elements
// [k * chunk, (k + 1) * chunk), which covers one or more row segments, and writes one partial per
// segment. Pure streaming: no atomics, nothing waits on another CTA.
template <typename T>
__global__ void __launch_bounds__(kThreads, 6)
sv_stats_kernel(const T *__restrict__ logits, int V, long long total, long long chunk, int maxseg,
                const RowInfo *__restrict__ rowinfo, StatPart *__restrict__ part,
                const unsigned *__restrict__ flags)
{
    if (flags[0]) return;
    const long long start = static_cast<long long>(blockIdx.x) * chunk;
    const long long stop = min(total, start + chunk);
    if (start >= stop) return;
    const int r_first = static_cast<int>(start / V);
    const int r_last = static_cast<int>((stop - 1) / V);
    for (int row = r_first; row <= r_last; ++row) {
        const long long rbase = static_cast<long long>(row) * V;
        const int b = static_cast<int>(max(start, rbase) - rbase);
        const int e = static_cast<int>(min(stop, rbase + V) - rbase);
        const int fk = static_cast<int>(rbase / chunk);
        stats_segment<T>(logits, V, row, b, e, static_cast<int>(blockIdx.x) - fk, maxseg, rowinfo,
                         part);
    }
}

// One warp per row: combine the row's segment partials in segment order (deterministic) and
// finalise it (acceptance test, race seeds, request completion).
template <typename T>
__global__ void __launch_bounds__(kThreads)
sv_finalize_kernel(const T *__restrict__ logits, int V, int rows, long long chunk, int maxseg,
                   const RowInfo *__restrict__ rowinfo, const StatPart *__restrict__ part,
                   const int32_t *__restrict__ draft_ids, const float *__restrict__ q,
                   uint64_t seed, uint32_t req_base, StatsOut o, const unsigned *__restrict__ flags)
{
    if (flags[0]) return;
    const int row = blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5);
    if (row >= rows) return;
    const int lane = threadIdx.x & 31;
    const RowInfo ri = rowinfo[row];
    const float c = ri.invT * kLog2e;
    const long long rbase = static_cast<long long>(row) * V;
    const int nseg = static_cast<int>((rbase + V - 1) / chunk) - static_cast<int>(rbase / chunk) + 1;
    float L = -kInf, s = 0.0f;
    int idx = INT_MAX;
    for (int k = lane; k < nseg; k += 32) {
        const float4 raw = __ldg(reinterpret_cast<const float4 *>(part) +
                                 static_cast<size_t>(row) * maxseg + k);
        combine_stat(L, s, idx, raw.x, raw.y, __float_as_int(raw.z), c);
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) {
        const float L2 = __shfl_xor_sync(0xFFFFFFFFu, L, o2);
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o2);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, idx, o2);
        combine_stat(L, s, idx, L2, s2, i2, c);
    }
    if (lane == 0)
        finalize_row<T>(logits + rbase, V, row, ri, L, s, idx, draft_ids, q, seed, req_base, o);
}

// ---------------------------------------------------------------------------------------
// Bulk-copy (TMA) staging: cp.async.bulk global -> shared, completion on an mbarrier. Every
// wait is bounded by the global timer.
// ---------------------------------------------------------------------------------------
constexpr unsigned long long kWaitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes) : "memory");
}
// Copy [src, src + bytes) to dst (both 16-byte aligned, bytes a multiple of 16), completing
// `bytes` of the transaction the barrier expects.
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}
__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}
// Wait for the phase with parity `parity`; false after `limit_ns` (never expected: the caller
// records an error and stops using the buffers).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, unsigned long long limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// ---------------------------------------------------------------------------------------
// 3. race + emit
// ---------------------------------------------------------------------------------------
// Screening. A thread skips a token only when its key is certainly below `ks`, a key that some
// candidate of the same race has already reached (so ks never exceeds the winner's key, and the
// winner -- or an equal key at a lower index -- is never skipped). ks is shared by the warp
// (redux), the CTA (shared memory) and all CTAs of the request (a global word).
struct RaceState {
    float kb = -kInf;        // this thread's best key
    int ib = -1;             // its index (-1: none yet)
    unsigned ks_enc = kKeyNone;
    float pre_x;             // p-race: skip a group whose max x is below this
    float kbl;               // p-race: (ks - delta) * log2 e
    float pre_rr;            // residual: skip a group whose rr upper bounds are all below this
    float ekb;               // residual: >= exp(delta - ks)
};

constexpr float kSafe = 1.0f + 0x1p-10f;  // covers MUFU and argument rounding errors

// Screening constants from ks. With delta = 1e-3 + 1e-5 |ks| (far above the few-ulp error of
// the binary32 key), a token whose key is certainly below ks - delta is skipped:
//   - with no randomness: key <= log w - log(clock) < log w + kClockLogMax;
//   - with its block's head: every clock of the block is >= E_min = -log(W)/16 >= (1 - W)/16,
//     so key < ks - delta once (1 - W)/16 > w exp(delta - ks);
//   - with its own slot word: clock >= (1 - W)/16 + (1 - U) (the slot a: (1 - W)/16).
__device__ __forceinline__ void refresh(RaceState &st)
{
    if (st.ks_enc == kKeyNone) {
        st.pre_x = -kInf;
        st.kbl = -kInf;
        st.pre_rr = -kInf;
        st.ekb = kInf;
        return;
    }
    const float ks = key_dec(st.ks_enc);
    const float delta = 1e-3f + 1e-5f * fabsf(ks);
    st.pre_x = ks - (sv::kClockLogMax + delta);
    st.kbl = (ks - delta) * kLog2e;
    st.pre_rr = sv::ex2_approx((ks - sv::kClockLogMax - delta) * kLog2e) * (1.0f - 0x1p-9f);
    st.ekb = sv::ex2_approx((delta - ks) * kLog2e) * kSafe;
}

__device__ __forceinline__ void raise_threshold(RaceState &st, unsigned enc)
{
    if (enc > st.ks_enc) {
        st.ks_enc = enc;
        refresh(st);
    }
}

__device__ __forceinline__ bool race_better(float ka, int ia, float kb, int ib)
{
    // is (ka, ia) better than (kb, ib)? larger key, then lower index; -1 = no candidate
    if (ia < 0) return false;
    if (ib < 0) return true;
    return ka > kb || (ka == kb && ia < ib);
}

// The full key out of line (rarely reached). NaN = not a candidate.
template <bool kResidual>
__device__ __noinline__ float race_key_slow(float x, float qv, uint32_t w_head, int a, int s,
                                            uint32_t w_slot, float m, float S)
{
    float key;
    const float E = race_clock(w_head, a, s, w_slot);
    return race_key<kResidual>(x, qv, E, m, S, key) ? key : __int_as_float(0x7FC00000);
}

// Offer token v (slot s of its block) whose clock is at least clock_lb; the full key is computed
// only if the screen cannot rule the token out. Returns true if the thread's threshold rose.
template <bool kResidual>
__device__ __forceinline__ bool race_offer(RaceState &st, unsigned *s_thr, int v, float x,
                                           float qv, float clock_lb, uint32_t w_head, int a,
                                           int s, uint32_t w_slot, float m, float S, float rr_up)
{
    if constexpr (kResidual) {
        if (!(rr_up > 0.0f)) return false;
        if (clock_lb > rr_up * st.ekb) return false;
    } else {
        if (clock_lb > sv::ex2_approx(fmaf(x, kLog2e, -st.kbl)) * kSafe) return false;
    }
    const float key = race_key_slow<kResidual>(x, qv, w_head, a, s, w_slot, m, S);
    if (key != key) return false;
    if (st.ib < 0 || key > st.kb) {
        st.kb = key;
        st.ib = v;
    }
    const unsigned enc = key_enc(key);
    if (enc > st.ks_enc) {
        raise_threshold(st, enc);
        atomicMax(s_thr, enc);
        return true;
    }
    return false;
}

__device__ __forceinline__ unsigned ld_relaxed(const unsigned *p)
{
    unsigned v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// One step of the race for this lane's 4 consecutive tokens v0..v0+3 (raw logit words lc, q words
// qc). The 4 lanes of a quad cover one 16-token clock block. Per block: the bound without
// randomness; then the quad's first lane draws the block head and the block is ruled out if even
// its smallest clock cannot beat ks; only then does each lane draw its own slots' words. Must be
// called by all 32 lanes of the warp (shuffles); lanes past the end pass v0 >= e. Returns true
// if this lane raised its threshold with a key of its own.
template <typename T, bool kResidual>
__device__ __forceinline__ bool race_step(RaceState &st, unsigned *s_thr,
                                          const uint32_t (&lc)[sizeof(T)], const uint32_t (&qc)[4],
                                          int v0, int e, float invT, float m, float S, int exclude,
                                          uint32_t j, uint32_t ireq, uint32_t k0, uint32_t k1)
{
    const int lane = threadIdx.x & 31;
    const int quarter = lane & 3;  // this lane's slots in the block: 4 * quarter .. 4 * quarter + 3
    float x[4], wv[4];  // x = logit / T; wv: the weight proxy the screens compare
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float l;
        if constexpr (sizeof(T) == 2)
            l = (k & 1) ? __uint_as_float(lc[k >> 1] & 0xFFFF0000u) : __uint_as_float(lc[k >> 1] << 16);
        else
            l = __uint_as_float(lc[k]);
        x[k] = __fmul_rn(l, invT);
        if constexpr (kResidual) {  // upper bound of rr = fma(-S, q, exp(x - m))
            const float t_up = sv::ex2_approx((x[k] - m) * kLog2e) * kSafe;
            wv[k] = v0 + k < e ? fmaf(-S, __uint_as_float(qc[k]), t_up) : -kInf;
        } else {
            wv[k] = v0 + k < e ? x[k] : -kInf;
        }
    }
    float mx = fmaxf(fmaxf(wv[0], wv[1]), fmaxf(wv[2], wv[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));  // the block's largest weight
    bool go;
    if (kResidual) go = (mx > 0.0f) && !(mx < st.pre_rr);
    else go = (mx > -kInf) && !(mx < st.pre_x);
    const uint32_t g = static_cast<uint32_t>(v0 - 4 * quarter) >> 4;
    uint32_t hw0 = 0u, hw1 = 0u;  // block head, drawn by the quad's first lane
    if (go && quarter == 0) {
        const sv::Philox4 h = sv::philox4x32_10(g, j, ireq, sv::kClockHead, k0, k1);
        hw0 = h.x;
        hw1 = h.y;
    }
    hw0 = __shfl_sync(0xFFFFFFFFu, hw0, lane & ~3);
    hw1 = __shfl_sync(0xFFFFFFFFu, hw1, lane & ~3);
    const float emin_lb = (1.0f - sv::uniform_from_word(hw0)) * 0.0625f;  // exact
    if (go) {
        const float cmax = kResidual ? mx * st.ekb
                                     : sv::ex2_approx(fmaf(mx, kLog2e, -st.kbl)) * kSafe;
        go = !(emin_lb > cmax);
    }
    bool raised = false;
    if (go) {
        const int a = static_cast<int>(hw1 & 15u);
        const sv::Philox4 r = sv::philox4x32_10(g, j, ireq, sv::kClockHead + 1u + quarter, k0, k1);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int v = v0 + k;
            if (v >= e || v == exclude) continue;
            const int s = 4 * quarter + k;
            const uint32_t ws = pick_word(r, k);
            const float lb = s == a ? emin_lb : emin_lb + (1.0f - sv::uniform_from_word(ws));
            raised |= race_offer<kResidual>(st, s_thr, v, x[k], __uint_as_float(qc[k]), lb, hw0,
                                            a, s, ws, m, S, wv[k]);
        }
    }
    return raised;
}

// Bring in the thresholds others have reached: the CTA's shared word every step, the request's
// global word every 4th step, read one exchange ahead (a stale value is a lower key and only
// screens less). After the step the warp shares its best threshold with one redux.
__device__ __forceinline__ void pull_threshold(RaceState &st, unsigned *s_thr, unsigned *g_thr,
                                               int step, unsigned &g_seen)
{
    raise_threshold(st, *reinterpret_cast<volatile unsigned *>(s_thr));
    if (g_thr && (step & 3) == 0) {
        if (g_seen > st.ks_enc) {
            raise_threshold(st, g_seen);
            atomicMax(s_thr, g_seen);
        }
        g_seen = ld_relaxed(g_thr);
    }
}

__device__ __forceinline__ void push_threshold(RaceState &st, unsigned *g_thr, bool raised)
{
    if (raised && g_thr) atomicMax(g_thr, st.ks_enc);  // publish to the other CTAs
    raise_threshold(st, __reduce_max_sync(0xFFFFFFFFu, st.ks_enc));  // share in the warp
}

template <typename T, bool kResidual>
__device__ __forceinline__ void load_quad(uint32_t (&l)[sizeof(T)], uint32_t (&qq)[4],
                                          const T *__restrict__ rp, const float *__restrict__ qrow,
                                          int v0, int e, bool aligned)
{
    if (aligned && v0 + 4 <= e) {
        if constexpr (sizeof(T) == 2) {
            const uint2 w = __ldg(reinterpret_cast<const uint2 *>(rp + v0));
            l[0] = w.x;
            l[1] = w.y;
        } else {
            const uint4 w = ldg_v4(rp + v0);
            l[0] = w.x; l[1] = w.y; l[2] = w.z; l[3] = w.w;
        }
        if constexpr (kResidual) {
            const uint4 w = ldg_v4(qrow + v0);
            qq[0] = w.x; qq[1] = w.y; qq[2] = w.z; qq[3] = w.w;
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const bool in = v0 + k < e;
            if constexpr (sizeof(T) == 2) {
                const uint32_t h = in ? static_cast<uint32_t>(__ldg(reinterpret_cast<const uint16_t *>(rp) + v0 + k)) : 0xFF80u;
                if (k & 1) l[k >> 1] |= h << 16;
                else l[k >> 1] = h;
            } else {
                l[k] = in ? __float_as_uint(__ldg(reinterpret_cast<const float *>(rp) + v0 + k)) : 0xFF800000u;
            }
            if constexpr (kResidual) qq[k] = in ? __float_as_uint(__ldg(qrow + v0 + k)) : 0u;
        }
    }
}

// Race over [b, e) of one row (b a multiple of 16) reading the logits (and q) directly from global
// memory, each thread with its next 4 tokens' loads in flight.
template <typename T, bool kResidual>
__device__ __forceinline__ void race_span(RaceState &st, unsigned *s_thr, unsigned *g_thr,
                                          const T *__restrict__ rp,
                                          const float *__restrict__ qrow, int b, int e,
                                          float invT, float m, float S, int exclude, uint32_t j,
                                          uint32_t ireq, uint32_t k0, uint32_t k1, bool aligned)
{
    constexpr int kStride = 4 * kThreads;
    uint32_t lc[sizeof(T)], ln[sizeof(T)], qc[4] = {0u, 0u, 0u, 0u}, qn[4] = {0u, 0u, 0u, 0u};
    unsigned g_seen = kKeyNone;
    const int warp_first = b + 4 * static_cast<int>(threadIdx.x & ~31u);
    int v0 = b + 4 * static_cast<int>(threadIdx.x);
    if (v0 < e) load_quad<T, kResidual>(lc, qc, rp, qrow, v0, e, aligned);
    int step = 0;
    for (int wf = warp_first; wf < e; wf += kStride, v0 += kStride, ++step) {
        if (v0 + kStride < e) load_quad<T, kResidual>(ln, qn, rp, qrow, v0 + kStride, e, aligned);
        pull_threshold(st, s_thr, g_thr, step, g_seen);
        const bool raised = race_step<T, kResidual>(st, s_thr, lc, qc, v0, e, invT, m, S, exclude,
                                                    j, ireq, k0, k1);
        push_threshold(st, g_thr, raised);
#pragma unroll
        for (int k = 0; k < static_cast<int>(sizeof(T)); ++k) lc[k] = ln[k];
#pragma unroll
        for (int k = 0; k < 4; ++k) qc[k] = qn[k];
    }
}

// Block reduction of (key, idx); result valid in thread 0.
__device__ __forceinline__ void block_reduce_race(float &kb, int &ib)
{
    __shared__ float sh_k[kThreads / 32];
    __shared__ int sh_i[kThreads / 32];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float k2 = __shfl_xor_sync(0xFFFFFFFFu, kb, o);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, ib, o);
        if (race_better(k2, i2, kb, ib)) {
            kb = k2;
            ib = i2;
        }
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();  // sh_* may still be read by a previous reduction
    if (lane == 0) {
        sh_k[warp] = kb;
        sh_i[warp] = ib;
    }
    __syncthreads();
    if (warp == 0) {
        kb = lane < kThreads / 32 ? sh_k[lane] : -kInf;
        ib = lane < kThreads / 32 ? sh_i[lane] : -1;
#pragma unroll
        for (int o = 4; o > 0; o >>= 1) {
            const float k2 = __shfl_xor_sync(0xFFFFFFFFu, kb, o);
            const int i2 = __shfl_xor_sync(0xFFFFFFFFu, ib, o);
            if (race_better(k2, i2, kb, ib)) {
                kb = k2;
                ib = i2;
            }
        }
    }
}

// Race over [b, e) of one row by the whole CTA. s_thr: the CTA's shared threshold word, set by
// the caller before a __syncthreads; g_thr: the request's global threshold word or nullptr.
template <typename T>
__device__ void race_row(float &kb, int &ib, unsigned *s_thr, unsigned *g_thr, const T *rp,
                         const float *qrow, int b, int e, float invT, float m, float S,
                         int exclude, uint32_t j, uint32_t ireq, uint64_t seed, bool aligned)
{
    RaceState st;
    refresh(st);
    const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    if (qrow)
        race_span<T, true>(st, s_thr, g_thr, rp, qrow, b, e, invT, m, S, exclude, j, ireq, k0, k1,
                           aligned);
    else
        race_span<T, false>(st, s_thr, g_thr, rp, qrow, b, e, invT, m, S, exclude, j, ireq, k0, k1,
                            aligned);
    kb = st.kb;
    ib = st.ib;
    block_reduce_race(kb, ib);
}

// The raced rows of all sampling requests, concatenated and split evenly over the CTAs. Each
// row occupies Vp = V rounded up to a multiple of 16 elements of that concatenation, so that
// every segment starts on a clock-block boundary within its row; a CTA whose segment lies in
// the padding publishes an empty partial.
template <typename T>
__global__ void __launch_bounds__(kThreads, 3)
sv_race_kernel(const T *__restrict__ logits, int V, int chunk_fixed, int maxseg,
               const ReqState *__restrict__ reqstate, const int *__restrict__ rand_req,
               const int *__restrict__ n_rand, const int32_t *__restrict__ draft_ids,
               const float *__restrict__ q, uint64_t seed, uint32_t req_base,
               RacePart *__restrict__ part, unsigned *__restrict__ race_counter,
               unsigned *__restrict__ race_thr, int32_t *__restrict__ sampled, int stride,
               int32_t *__restrict__ num_sampled, int32_t *__restrict__ num_rejected,
               const unsigned *__restrict__ flags, bool aligned)
{
    if (flags[0]) return;
    const int Vp = (V + 15) & ~15;
    const long long total = static_cast<long long>(*n_rand) * Vp;
    long long chunk = chunk_fixed;
    if (chunk <= 0) {
        chunk = (total + gridDim.x - 1) / gridDim.x;
        chunk = max((chunk + 15) / 16 * 16, static_cast<long long>(kMinChunk));
    }
    const long long start = static_cast<long long>(blockIdx.x) * chunk;
    const long long stop = min(total, start + chunk);
    if (start >= stop) return;

    __shared__ unsigned s_thr;
    __shared__ int s_last, s_token;
    const int vr_first = static_cast<int>(start / Vp);
    const int vr_last = static_cast<int>((stop - 1) / Vp);
    for (int vr = vr_first; vr <= vr_last; ++vr) {
        const long long vbase = static_cast<long long>(vr) * Vp;
        const int b = static_cast<int>(max(start, vbase) - vbase);
        const int e = static_cast<int>(min(min(stop, vbase + Vp) - vbase, static_cast<long long>(V)));
        const int fk = static_cast<int>(vbase / chunk);
        const int nseg = static_cast<int>((vbase + Vp - 1) / chunk) - fk + 1;
        const int seg = static_cast<int>(blockIdx.x) - fk;
        const int i = rand_req[vr];
        const ReqState rq = reqstate[i];
        const T *rp = logits + static_cast<size_t>(rq.row) * static_cast<size_t>(V);
        const float *qrow = (rq.jstar < rq.K && q) ? q + static_cast<size_t>(rq.q0 + rq.jstar) * V
                                                   : nullptr;
        const uint32_t ireq = req_base + static_cast<uint32_t>(i);
        if (threadIdx.x == 0) s_thr = rq.seed;  // the argmax token's key seeds the threshold
        __syncthreads();
        float kb;
        int ib;
        race_row<T>(kb, ib, &s_thr, &race_thr[i], rp, qrow, b, e, rq.invT, rq.m, rq.S, rq.excl,
                    static_cast<uint32_t>(rq.jstar), ireq, seed, aligned);
        if (nseg > 1) {
            if (threadIdx.x == 0) {
                part[static_cast<size_t>(i) * maxseg + seg] = RacePart{kb, ib};
                __threadfence();
                const unsigned ticket = atomicAdd(&race_counter[i], 1u);
                s_last = ticket == static_cast<unsigned>(nseg - 1);
            }
            __syncthreads();
            if (!s_last) continue;
            __threadfence();
            if (threadIdx.x < 32) {
                float kw = -kInf;
                int iw = -1;
                for (int k = threadIdx.x; k < nseg; k += 32) {
                    const float2 raw = __ldcg(reinterpret_cast<const float2 *>(part) +
                                              static_cast<size_t>(i) * maxseg + k);
                    const int i2 = __float_as_int(raw.y);
                    if (race_better(raw.x, i2, kw, iw)) {
                        kw = raw.x;
                        iw = i2;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float k2 = __shfl_xor_sync(0xFFFFFFFFu, kw, o);
                    const int i2 = __shfl_xor_sync(0xFFFFFFFFu, iw, o);
                    if (race_better(k2, i2, kw, iw)) {
                        kw = k2;
                        iw = i2;
                    }
                }
                if (threadIdx.x == 0) {
                    ib = iw;
                    race_counter[i] = 0u;
                }
            }
        }
        if (threadIdx.x == 0) s_token = ib;
        __syncthreads();
        int token = s_token;
        if (token < 0) {
            // Nothing left after rounding (residual with p <= q everywhere, or V == 1 with the
            // only token excluded): draw from p itself so the output stays a target-side draw.
            if (threadIdx.x == 0) s_thr = rq.seed_p;
            __syncthreads();
            race_row<T>(kb, ib, &s_thr, nullptr, rp, nullptr, 0, V, rq.invT, rq.m, rq.S, -1,
                        static_cast<uint32_t>(rq.jstar), ireq, seed, aligned);
            if (threadIdx.x == 0) s_token = ib;
            __syncthreads();
            token = s_token;
        }
        emit_row(i, rq.jstar, rq.K, rq.q0, token, draft_ids, sampled, stride, num_sampled,
                 num_rejected, threadIdx.x, kThreads);
        __syncthreads();  // s_thr / s_token are reused by the next row of this CTA
    }
}


// ---------------------------------------------------------------------------------------
// Race with the raced rows staged through shared memory: same partition and results as
// sv_race_kernel, for rows that start on 16-byte boundaries. The CTA's segments are cut into
// stages of up to kRaceStageTok tokens (never crossing a row); one thread issues bulk copies of
// each stage's logits and q into a ring of kRaceStages buffers, so that several stages per CTA
// are in flight while the warps screen the current one from shared memory.
// ---------------------------------------------------------------------------------------
constexpr int kRaceStageTok = 2048;
constexpr int kRaceStages = 4;
template <typename T> __host__ __device__ constexpr int race_stage_bytes() { return kRaceStageTok * (static_cast<int>(sizeof(T)) + 4); }

// Segment of virtual row vr inside [start, stop): token range [b, e) of the real row.
struct RaceSeg {
    int b, e;
};
__device__ __forceinline__ RaceSeg race_seg(int vr, int Vp, int V, long long start, long long stop)
{
    const long long vbase = static_cast<long long>(vr) * Vp;
    const int b = static_cast<int>(max(start, vbase) - vbase);
    const int e = static_cast<int>(min(min(stop, vbase + Vp) - vbase, static_cast<long long>(V)));
    return RaceSeg{b, max(b, e)};
}

template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
sv_race_bulk_kernel(const T *__restrict__ logits, int V, int chunk_fixed, int maxseg,
                    const ReqState *__restrict__ reqstate, const int *__restrict__ rand_req,
                    const int *__restrict__ n_rand, const int32_t *__restrict__ draft_ids,
                    const float *__restrict__ q, uint64_t seed, uint32_t req_base,
                    RacePart *__restrict__ part, unsigned *__restrict__ race_counter,
                    unsigned *__restrict__ race_thr, int32_t *__restrict__ sampled, int stride,
                    int32_t *__restrict__ num_sampled, int32_t *__restrict__ num_rejected,
                    unsigned *__restrict__ flags)
{
    extern __shared__ __align__(128) unsigned char ring[];
    __shared__ __align__(8) uint64_t full[kRaceStages];
    __shared__ unsigned s_thr;
    __shared__ int s_last, s_token, s_abort;
    if (flags[0]) return;
    const int Vp = (V + 15) & ~15;
    const long long total = static_cast<long long>(*n_rand) * Vp;
    long long chunk = chunk_fixed;
    if (chunk <= 0) {
        chunk = (total + gridDim.x - 1) / gridDim.x;
        chunk = max((chunk + 15) / 16 * 16, static_cast<long long>(kMinChunk));
    }
    const long long start = static_cast<long long>(blockIdx.x) * chunk;
    const long long stop = min(total, start + chunk);
    if (start >= stop) return;
    const int vr_first = static_cast<int>(start / Vp);
    const int vr_last = static_cast<int>((stop - 1) / Vp);
    constexpr int kStageBytes = race_stage_bytes<T>();
    constexpr int kQOff = kRaceStageTok * static_cast<int>(sizeof(T));  // q part of a stage

    // producer (thread 0): walks the same stage sequence as the consumers, ahead of them
    int p_vr = vr_first, p_tok = 0, p_end = 0, issued = 0;
    const T *p_rp = nullptr;
    const float *p_q = nullptr;
    auto p_enter_row = [&]() {  // position the producer at the first stage of row p_vr
        while (p_vr <= vr_last) {
            const RaceSeg sg = race_seg(p_vr, Vp, V, start, stop);
            if (sg.b < sg.e) {
                const ReqState rq = reqstate[rand_req[p_vr]];
                p_rp = logits + static_cast<size_t>(rq.row) * static_cast<size_t>(V);
                p_q = (rq.jstar < rq.K && q) ? q + static_cast<size_t>(rq.q0 + rq.jstar) * V : nullptr;
                p_tok = sg.b;
                p_end = sg.e;
                return;
            }
            ++p_vr;
        }
    };
    auto p_issue = [&](int buf) {  // issue the next stage into ring buffer buf, if any
        if (p_vr > vr_last) return;
        const int n = min(kRaceStageTok, p_end - p_tok);
        const uint32_t lb = static_cast<uint32_t>(n) * sizeof(T);
        const uint32_t qb = p_q ? static_cast<uint32_t>(n) * 4u : 0u;
        unsigned char *dst = ring + buf * kStageBytes;
        mbar_expect(&full[buf], lb + qb);
        bulk_load(dst, p_rp + p_tok, lb, &full[buf]);
        if (qb) bulk_load(dst + kQOff, p_q + p_tok, qb, &full[buf]);
        ++issued;
        p_tok += n;
        if (p_tok >= p_end) {
            ++p_vr;
            p_enter_row();
        }
    };
    if (threadIdx.x == 0) {
        for (int b2 = 0; b2 < kRaceStages; ++b2) mbar_init(&full[b2], 1);
        mbar_fence_init();
        s_abort = 0;
        p_enter_row();
        for (int b2 = 0; b2 < kRaceStages; ++b2) p_issue(b2);
    }
    __syncthreads();

    const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    int k = 0;  // consumer's stage counter
    bool aborted = false;
    for (int vr = vr_first; vr <= vr_last && !aborted; ++vr) {
        const RaceSeg sg = race_seg(vr, Vp, V, start, stop);
        const long long vbase = static_cast<long long>(vr) * Vp;
        const int fk = static_cast<int>(vbase / chunk);
        const int nseg = static_cast<int>((vbase + Vp - 1) / chunk) - fk + 1;
        const int seg = static_cast<int>(blockIdx.x) - fk;
        const int i = rand_req[vr];
        const ReqState rq = reqstate[i];
        const bool residual = rq.jstar < rq.K && q != nullptr;
        const uint32_t ireq = req_base + static_cast<uint32_t>(i);
        const uint32_t j = static_cast<uint32_t>(rq.jstar);
        if (threadIdx.x == 0) s_thr = rq.seed;  // the argmax token's key seeds the threshold
        __syncthreads();
        RaceState st;
        refresh(st);
        unsigned g_seen = kKeyNone;
        int step = 0;
        for (int t0 = sg.b; t0 < sg.e; t0 += kRaceStageTok, ++k) {
            const int n = min(kRaceStageTok, sg.e - t0);
            const int buf = k % kRaceStages;
            if (!mbar_wait(&full[buf], static_cast<uint32_t>(k / kRaceStages) & 1u, kWaitNs)) {
                s_abort = 1;
                atomicOr(&flags[1], SV_ERR_TIMEOUT);
            }
            const unsigned char *stage = ring + buf * kStageBytes;
            for (int pass = 0; pass * 4 * kThreads < n; ++pass, ++step) {
                const int tl = pass * 4 * kThreads + 4 * static_cast<int>(threadIdx.x);  // in stage
                uint32_t lc[sizeof(T)], qc[4] = {0u, 0u, 0u, 0u};
                if (tl < n) {
                    if constexpr (sizeof(T) == 2) {
                        const uint2 w = *reinterpret_cast<const uint2 *>(stage + tl * 2);
                        lc[0] = w.x;
                        lc[1] = w.y;
                    } else {
                        const uint4 w = *reinterpret_cast<const uint4 *>(stage + tl * 4);
                        lc[0] = w.x; lc[1] = w.y; lc[2] = w.z; lc[3] = w.w;
                    }
                    if (residual) {
                        const uint4 w = *reinterpret_cast<const uint4 *>(stage + kQOff + tl * 4);
                        qc[0] = w.x; qc[1] = w.y; qc[2] = w.z; qc[3] = w.w;
                    }
                } else {
#pragma unroll
                    for (int h = 0; h < static_cast<int>(sizeof(T)); ++h) lc[h] = 0xFF80FF80u;
                }
                pull_threshold(st, &s_thr, &race_thr[i], step, g_seen);
                bool raised;
                if (residual)
                    raised = race_step<T, true>(st, &s_thr, lc, qc, t0 + tl, sg.e, rq.invT, rq.m,
                                                rq.S, rq.excl, j, ireq, k0, k1);
                else
                    raised = race_step<T, false>(st, &s_thr, lc, qc, t0 + tl, sg.e, rq.invT, rq.m,
                                                 rq.S, rq.excl, j, ireq, k0, k1);
                push_threshold(st, &race_thr[i], raised);
            }
            __syncthreads();  // every thread is done with this buffer
            if (s_abort) {
                aborted = true;
                break;
            }
            if (threadIdx.x == 0) {
                fence_proxy_async_smem();
                p_issue(buf);
            }
        }
        if (aborted) break;
        float kb = st.kb;
        int ib = st.ib;
        block_reduce_race(kb, ib);
        if (nseg > 1) {
            if (threadIdx.x == 0) {
                part[static_cast<size_t>(i) * maxseg + seg] = RacePart{kb, ib};
                __threadfence();
                const unsigned ticket = atomicAdd(&race_counter[i], 1u);
                s_last = ticket == static_cast<unsigned>(nseg - 1);
            }
            __syncthreads();
            if (!s_last) continue;
            __threadfence();
            if (threadIdx.x < 32) {
                float kw = -kInf;
                int iw = -1;
                for (int kk = threadIdx.x; kk < nseg; kk += 32) {
                    const float2 raw = __ldcg(reinterpret_cast<const float2 *>(part) +
                                              static_cast<size_t>(i) * maxseg + kk);
                    const int i2 = __float_as_int(raw.y);
                    if (race_better(raw.x, i2, kw, iw)) {
                        kw = raw.x;
                        iw = i2;
                    }
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) {
                    const float k2 = __shfl_xor_sync(0xFFFFFFFFu, kw, o);
                    const int i2 = __shfl_xor_sync(0xFFFFFFFFu, iw, o);
                    if (race_better(k2, i2, kw, iw)) {
                        kw = k2;
                        iw = i2;
                    }
                }
                if (threadIdx.x == 0) {
                    ib = iw;
                    race_counter[i] = 0u;
                }
            }
        }
        if (threadIdx.x == 0) s_token = ib;
        __syncthreads();
        int token = s_token;
        if (token < 0) {
            // nothing left of the residual after rounding: draw from p itself (global reads)
            const T *rp = logits + static_cast<size_t>(rq.row) * static_cast<size_t>(V);
            if (threadIdx.x == 0) s_thr = rq.seed_p;
            __syncthreads();
            race_row<T>(kb, ib, &s_thr, nullptr, rp, nullptr, 0, V, rq.invT, rq.m, rq.S, -1, j,
                        ireq, seed, true);
            if (threadIdx.x == 0) s_token = ib;
            __syncthreads();
            token = s_token;
        }
        emit_row(i, rq.jstar, rq.K, rq.q0, token, draft_ids, sampled, stride, num_sampled,
                 num_rejected, threadIdx.x, kThreads);
        __syncthreads();  // s_thr / s_token are reused by the next row of this CTA
    }
    if (aborted && threadIdx.x == 0) {
        // let the copies still in flight land before the CTA's shared memory is released
        for (int kk = k + 1; kk < issued; ++kk)
            mbar_wait(&full[kk % kRaceStages], static_cast<uint32_t>(kk / kRaceStages) & 1u, kWaitNs / 4);
    }
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
constexpr int kProfRing = 512;

constexpr int kKernels = 4;  // plan, stats, finalize, race

struct ProfSlot {
    cudaEvent_t ev[kKernels + 1];
    bool pending;
};

int round_up8(int x) { return (x + 7) / 8 * 8; }
int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

struct spec_verify_ctx {
    int device = 0;
    int max_num_reqs = 0, max_spec_len = 0, V = 0, dtype = SV_F32, has_q = 0;
    int max_rows = 0, maxseg = 0;
    int stats_chunk = 0, race_chunk = 0;  // 0: automatic (even split over the grid)
    int stats_ctas = 1, race_ctas = 1;    // one wave of each kernel (SMs x CTAs per SM)
    int race_bulk_ctas = 1;
    RowInfo *rowinfo = nullptr;
    RowStat *rowstat = nullptr;
    StatPart *statpart = nullptr;
    ReqState *reqstate = nullptr;
    RacePart *racepart = nullptr;
    // [N] rows done | [N] race counters | [N] race thresholds | [N] sampling-request list |
    // [1] its length
    unsigned *counters = nullptr;
    unsigned *flags = nullptr;  // [0] per-call batch-invalid, [1] sticky error word
    // host-buffer staging
    void *io_logits = nullptr;
    float *io_q = nullptr;
    int32_t *io_small = nullptr;  // ids | cu | sampled | num_sampled | num_rejected
    float *io_temp = nullptr;
    uint8_t *io_greedy = nullptr;
    // profiling
    bool prof = false;
    std::vector<ProfSlot> ring;
    int64_t prof_calls = 0, prof_done = 0;
    double prof_ms[kKernels] = {0, 0, 0, 0};
};

namespace {

constexpr size_t counter_words(size_t reqs) { return 4 * reqs + 1; }

ReqWords req_words(spec_verify_ctx *ctx)
{
    unsigned *base = ctx->counters;
    const size_t N = static_cast<size_t>(ctx->max_num_reqs);
    return ReqWords{base, base + N, base + 2 * N, reinterpret_cast<int *>(base + 3 * N),
                    reinterpret_cast<int *>(base + 4 * N)};
}

struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            ok = false;
            return;
        }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

void prof_collect(spec_verify_ctx *ctx, ProfSlot &s)
{
    if (!s.pending) return;
    cudaEventSynchronize(s.ev[kKernels]);
    for (int k = 0; k < kKernels; ++k) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, s.ev[k], s.ev[k + 1]) == cudaSuccess) ctx->prof_ms[k] += ms;
    }
    s.pending = false;
    ctx->prof_done++;
}

void free_all(spec_verify_ctx *ctx)
{
    cudaFree(ctx->rowinfo);
    cudaFree(ctx->rowstat);
    cudaFree(ctx->statpart);
    cudaFree(ctx->reqstate);
    cudaFree(ctx->racepart);
    cudaFree(ctx->counters);
    cudaFree(ctx->flags);
    cudaFree(ctx->io_logits);
    cudaFree(ctx->io_q);
    cudaFree(ctx->io_small);
    cudaFree(ctx->io_temp);
    cudaFree(ctx->io_greedy);
    for (auto &s : ctx->ring)
        for (auto &e : s.ev) cudaEventDestroy(e);
    ctx->ring.clear();
}

// Allow the staged race its shared-memory ring and report how many CTAs of each kernel fit on
// one SM (for the one-wave grids).
template <typename T>
cudaError_t occupancy(int *stats_per_sm, int *race_per_sm, int *race_bulk_per_sm)
{
    cudaError_t e = cudaFuncSetAttribute(sv_race_bulk_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kRaceStages * race_stage_bytes<T>());
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(stats_per_sm, sv_stats_kernel<T>, kThreads, 0);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(race_bulk_per_sm, sv_race_bulk_kernel<T>,
                                                      kThreads, kRaceStages * race_stage_bytes<T>());
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(race_per_sm, sv_race_kernel<T>, kThreads, 0);
}

template <typename T>
int launch_all(spec_verify_ctx *ctx, const T *logits, const int32_t *draft_ids, const float *q,
               const int32_t *cu, const float *temperature, const uint8_t *is_greedy,
               uint64_t seed, uint32_t base, int num_reqs, int nd, int kmax, int32_t *sampled,
               int32_t *num_sampled, int32_t *num_rejected, float *opt_max, float *opt_sum,
               int32_t *opt_amax, cudaStream_t stream)
{
    const int V = ctx->V;
    const int rows = nd + num_reqs;
    const int stride = kmax + 1;
    const ReqWords rw = req_words(ctx);

    // statistics: the flattened [rows x V] logits split evenly over kStatsWaves waves
    const long long total = static_cast<long long>(rows) * V;
    long long chunk1 = ctx->stats_chunk;
    if (chunk1 <= 0) chunk1 = (total + kStatsWaves * ctx->stats_ctas - 1) / (kStatsWaves * ctx->stats_ctas);
    chunk1 = std::max<long long>((chunk1 + 7) / 8 * 8, kMinChunk);
    const int grid1 = static_cast<int>((total + chunk1 - 1) / chunk1);
    // Every row (and q row) starts on a 16-byte boundary when V is a multiple of 8 (bf16) or 4
    // (fp32); base pointers are checked to be 16-byte aligned: the race can use vector loads and
    // stage the rows through shared memory with bulk copies.
    const bool aligned = V % static_cast<int>(16 / sizeof(T)) == 0;
    // race: the raced rows (at most one per request) split evenly over kRaceWaves waves
    const int grid2 = ctx->race_chunk > 0
                          ? static_cast<int>((static_cast<long long>(num_reqs) * ((V + 15) & ~15) + ctx->race_chunk - 1) / ctx->race_chunk)
                          : kRaceWaves * (aligned ? ctx->race_bulk_ctas : ctx->race_ctas);
    const StatsOut so{ctx->rowstat, ctx->reqstate, rw.rows_done, sampled, num_sampled, num_rejected,
                      stride, opt_max, opt_sum, opt_amax};

    ProfSlot *slot = nullptr;
    if (ctx->prof) {
        slot = &ctx->ring[static_cast<size_t>(ctx->prof_calls % kProfRing)];
        prof_collect(ctx, *slot);
        cudaEventRecord(slot->ev[0], stream);
    }
    sv_plan_kernel<<<1, kPlanThreads, 0, stream>>>(cu, temperature, is_greedy, num_reqs, nd, kmax,
                                                   ctx->rowinfo, rw, sampled, stride, num_sampled,
                                                   num_rejected, ctx->flags);
    if (slot) cudaEventRecord(slot->ev[1], stream);
    sv_stats_kernel<T><<<grid1, kThreads, 0, stream>>>(logits, V, total, chunk1, ctx->maxseg,
                                                       ctx->rowinfo, ctx->statpart, ctx->flags);
    if (slot) cudaEventRecord(slot->ev[2], stream);
    sv_finalize_kernel<T><<<(rows + kThreads / 32 - 1) / (kThreads / 32), kThreads, 0, stream>>>(
        logits, V, rows, chunk1, ctx->maxseg, ctx->rowinfo, ctx->statpart, draft_ids, q, seed,
        base, so, ctx->flags);
    if (slot) cudaEventRecord(slot->ev[3], stream);
    if (aligned)
        sv_race_bulk_kernel<T><<<grid2, kThreads, kRaceStages * race_stage_bytes<T>(), stream>>>(
            logits, V, ctx->race_chunk, ctx->maxseg, ctx->reqstate, rw.rand_req, rw.n_rand,
            draft_ids, q, seed, base, ctx->racepart, rw.race_counter, rw.race_thr, sampled, stride,
            num_sampled, num_rejected, ctx->flags);
    else
        sv_race_kernel<T><<<grid2, kThreads, 0, stream>>>(
            logits, V, ctx->race_chunk, ctx->maxseg, ctx->reqstate, rw.rand_req, rw.n_rand,
            draft_ids, q, seed, base, ctx->racepart, rw.race_counter, rw.race_thr, sampled, stride,
            num_sampled, num_rejected, ctx->flags, aligned);
    if (slot) {
        cudaEventRecord(slot->ev[4], stream);
        slot->pending = true;
        ctx->prof_calls++;
    }
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

int check_run_args(const spec_verify_ctx *ctx, const void *logits, const int32_t *draft_ids,
                   const float *draft_probs, const int32_t *cu, const float *temperature,
                   const uint8_t *is_greedy, int num_reqs, int nd, int kmax,
                   const int32_t *sampled, const int32_t *num_sampled, const int32_t *num_rejected)
{
    if (num_reqs < 0 || nd < 0 || kmax < 0) return SV_EINVAL;
    if (num_reqs > ctx->max_num_reqs || kmax > ctx->max_spec_len ||
        static_cast<long long>(nd) > static_cast<long long>(num_reqs) * kmax)
        return SV_ECAPACITY;
    if (num_reqs == 0) return SV_OK;
    if (!logits || !cu || !temperature || !is_greedy || !sampled || !num_sampled ||
        !num_rejected || (nd > 0 && !draft_ids))
        return SV_EINVAL;
    if (draft_probs && !ctx->has_q) return SV_EINVAL;
    return SV_OK;
}

}  // namespace

extern "C" {

int spec_verify_init(spec_verify_ctx **out, int max_num_reqs, int max_spec_len, int vocab_size,
                     int logits_dtype, int has_draft_probs, int device)
{
    if (!out) return SV_EINVAL;
    *out = nullptr;
    if (max_num_reqs <= 0 || max_spec_len < 0 || vocab_size <= 0) return SV_EINVAL;
    if (logits_dtype != SV_F32 && logits_dtype != SV_BF16) return SV_EDTYPE;
    const long long rows = static_cast<long long>(max_num_reqs) * (max_spec_len + 1);
    const long long maxseg = ceil_div(vocab_size, kMinChunk) + 1;
    if (rows > INT_MAX / 8 || rows * maxseg > (1LL << 31) || static_cast<long long>(max_num_reqs) * maxseg > (1LL << 31))
        return SV_ECAPACITY;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) {
        cudaGetLastError();
        return SV_EDEVICE;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return SV_EDEVICE;
    if (prop.major != 10 || prop.minor != 3) return SV_EDEVICE;  // built for sm_103a only
    DeviceGuard g(device);
    if (!g.ok) return SV_EDEVICE;

    auto *ctx = new (std::nothrow) spec_verify_ctx();
    if (!ctx) return SV_ECAPACITY;
    ctx->device = device;
    ctx->max_num_reqs = max_num_reqs;
    ctx->max_spec_len = max_spec_len;
    ctx->V = vocab_size;
    ctx->dtype = logits_dtype;
    ctx->has_q = has_draft_probs != 0;
    ctx->max_rows = static_cast<int>(rows);
    ctx->maxseg = static_cast<int>(maxseg);
    const size_t R = static_cast<size_t>(rows), N = static_cast<size_t>(max_num_reqs);
    const size_t P = static_cast<size_t>(maxseg);
    const size_t W = counter_words(N);
    bool ok = cudaMalloc(&ctx->rowinfo, R * sizeof(RowInfo)) == cudaSuccess &&
              cudaMalloc(&ctx->rowstat, R * sizeof(RowStat)) == cudaSuccess &&
              cudaMalloc(&ctx->statpart, R * P * sizeof(StatPart)) == cudaSuccess &&
              cudaMalloc(&ctx->reqstate, N * sizeof(ReqState)) == cudaSuccess &&
              cudaMalloc(&ctx->racepart, N * P * sizeof(RacePart)) == cudaSuccess &&
              cudaMalloc(&ctx->counters, W * sizeof(unsigned)) == cudaSuccess &&
              cudaMalloc(&ctx->flags, 2 * sizeof(unsigned)) == cudaSuccess;
    ok = ok && cudaMemset(ctx->counters, 0, W * sizeof(unsigned)) == cudaSuccess &&
         cudaMemset(ctx->flags, 0, 2 * sizeof(unsigned)) == cudaSuccess;
    int stats_per_sm = 0, race_per_sm = 0, race_bulk_per_sm = 0;
    ok = ok && (logits_dtype == SV_BF16
                    ? occupancy<uint16_t>(&stats_per_sm, &race_per_sm, &race_bulk_per_sm)
                    : occupancy<float>(&stats_per_sm, &race_per_sm, &race_bulk_per_sm)) == cudaSuccess;
    ok = ok && cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
        free_all(ctx);
        delete ctx;
        cudaGetLastError();
        return SV_ECUDA;
    }
    ctx->stats_ctas = std::max(stats_per_sm, 1) * prop.multiProcessorCount;
    ctx->race_ctas = std::max(race_per_sm, 1) * prop.multiProcessorCount;
    ctx->race_bulk_ctas = std::max(race_bulk_per_sm, 1) * prop.multiProcessorCount;
    *out = ctx;
    return SV_OK;
}

int spec_verify_run(spec_verify_ctx *ctx, const void *logits, const int32_t *draft_ids,
                    const float *draft_probs, const int32_t *cu_num_draft,
                    const float *temperature, const uint8_t *is_greedy, uint64_t seed,
                    uint32_t req_index_base, int num_reqs, int num_draft_tokens,
                    int max_spec_len_this_batch, int32_t *sampled, int32_t *num_sampled,
                    int32_t *num_rejected, float *opt_row_max, float *opt_row_sumexp,
                    int32_t *opt_row_argmax, void *cuda_stream)
{
    if (!ctx) return SV_EINVAL;
    int rc = check_run_args(ctx, logits, draft_ids, draft_probs, cu_num_draft, temperature,
                            is_greedy, num_reqs, num_draft_tokens, max_spec_len_this_batch,
                            sampled, num_sampled, num_rejected);
    if (rc != SV_OK || num_reqs == 0) return rc;
    if (reinterpret_cast<uintptr_t>(logits) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(draft_probs) % 16 != 0)
        return SV_EINVAL;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
    auto stream = static_cast<cudaStream_t>(cuda_stream);
    if (ctx->dtype == SV_BF16)
        return launch_all<uint16_t>(ctx, static_cast<const uint16_t *>(logits), draft_ids,
                                    draft_probs, cu_num_draft, temperature, is_greedy, seed,
                                    req_index_base, num_reqs, num_draft_tokens,
                                    max_spec_len_this_batch, sampled, num_sampled, num_rejected,
                                    opt_row_max, opt_row_sumexp, opt_row_argmax, stream);
    return launch_all<float>(ctx, static_cast<const float *>(logits), draft_ids, draft_probs,
                             cu_num_draft, temperature, is_greedy, seed, req_index_base, num_reqs,
                             num_draft_tokens, max_spec_len_this_batch, sampled, num_sampled,
                             num_rejected, opt_row_max, opt_row_sumexp, opt_row_argmax, stream);
}

int spec_verify_reserve_host_io(spec_verify_ctx *ctx)
{
    if (!ctx) return SV_EINVAL;
    if (ctx->io_logits) return SV_OK;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
    const size_t R = static_cast<size_t>(ctx->max_rows), V = static_cast<size_t>(ctx->V);
    const size_t N = static_cast<size_t>(ctx->max_num_reqs);
    const size_t D = N * static_cast<size_t>(ctx->max_spec_len);
    const size_t eb = ctx->dtype == SV_BF16 ? 2 : 4;
    const size_t small = D + (N + 1) + N * (ctx->max_spec_len + 1) + 2 * N;
    bool ok = cudaMalloc(&ctx->io_logits, R * V * eb) == cudaSuccess &&
              (!ctx->has_q || D == 0 || cudaMalloc(&ctx->io_q, D * V * sizeof(float)) == cudaSuccess) &&
              cudaMalloc(&ctx->io_small, small * sizeof(int32_t)) == cudaSuccess &&
              cudaMalloc(&ctx->io_temp, N * sizeof(float)) == cudaSuccess &&
              cudaMalloc(&ctx->io_greedy, N) == cudaSuccess;
    if (!ok) {
        cudaFree(ctx->io_logits);
        cudaFree(ctx->io_q);
        cudaFree(ctx->io_small);
        cudaFree(ctx->io_temp);
        cudaFree(ctx->io_greedy);
        ctx->io_logits = nullptr;
        ctx->io_q = nullptr;
        ctx->io_small = nullptr;
        ctx->io_temp = nullptr;
        ctx->io_greedy = nullptr;
        cudaGetLastError();
        return SV_ECUDA;
    }
    return SV_OK;
}

int spec_verify_run_host(spec_verify_ctx *ctx, const void *logits, const int32_t *draft_ids,
                         const float *draft_probs, const int32_t *cu_num_draft,
                         const float *temperature, const uint8_t *is_greedy, uint64_t seed,
                         uint32_t req_index_base, int num_reqs, int num_draft_tokens,
                         int max_spec_len_this_batch, int32_t *sampled, int32_t *num_sampled,
                         int32_t *num_rejected, void *cuda_stream)
{
    if (!ctx) return SV_EINVAL;
    if (!ctx->io_logits) return SV_EINVAL;
    int rc = check_run_args(ctx, logits, draft_ids, draft_probs, cu_num_draft, temperature,
                            is_greedy, num_reqs, num_draft_tokens, max_spec_len_this_batch,
                            sampled, num_sampled, num_rejected);
    if (rc != SV_OK || num_reqs == 0) return rc;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
    auto stream = static_cast<cudaStream_t>(cuda_stream);
    const size_t V = static_cast<size_t>(ctx->V);
    const size_t eb = ctx->dtype == SV_BF16 ? 2 : 4;
    const size_t rows = static_cast<size_t>(num_draft_tokens) + num_reqs;
    const size_t N = static_cast<size_t>(ctx->max_num_reqs);
    const size_t D = N * static_cast<size_t>(ctx->max_spec_len);
    int32_t *d_ids = ctx->io_small;
    int32_t *d_cu = d_ids + D;
    int32_t *d_sampled = d_cu + (N + 1);
    int32_t *d_ns = d_sampled + N * (ctx->max_spec_len + 1);
    int32_t *d_nr = d_ns + N;
    const size_t stride = static_cast<size_t>(max_spec_len_this_batch) + 1;
    bool ok = cudaMemcpyAsync(ctx->io_logits, logits, rows * V * eb, cudaMemcpyHostToDevice, stream) == cudaSuccess &&
              (!draft_probs || cudaMemcpyAsync(ctx->io_q, draft_probs, static_cast<size_t>(num_draft_tokens) * V * 4,
                                               cudaMemcpyHostToDevice, stream) == cudaSuccess) &&
              (num_draft_tokens == 0 || cudaMemcpyAsync(d_ids, draft_ids, static_cast<size_t>(num_draft_tokens) * 4,
                                                        cudaMemcpyHostToDevice, stream) == cudaSuccess) &&
              cudaMemcpyAsync(d_cu, cu_num_draft, (static_cast<size_t>(num_reqs) + 1) * 4,
                              cudaMemcpyHostToDevice, stream) == cudaSuccess &&
              cudaMemcpyAsync(ctx->io_temp, temperature, static_cast<size_t>(num_reqs) * 4,
                              cudaMemcpyHostToDevice, stream) == cudaSuccess &&
              cudaMemcpyAsync(ctx->io_greedy, is_greedy, static_cast<size_t>(num_reqs),
                              cudaMemcpyHostToDevice, stream) == cudaSuccess;
    if (!ok) return SV_ECUDA;
    rc = spec_verify_run(ctx, ctx->io_logits, d_ids, draft_probs ? ctx->io_q : nullptr, d_cu,
                         ctx->io_temp, ctx->io_greedy, seed, req_index_base, num_reqs,
                         num_draft_tokens, max_spec_len_this_batch, d_sampled, d_ns, d_nr,
                         nullptr, nullptr, nullptr, cuda_stream);
    if (rc != SV_OK) return rc;
    ok = cudaMemcpyAsync(sampled, d_sampled, static_cast<size_t>(num_reqs) * stride * 4,
                         cudaMemcpyDeviceToHost, stream) == cudaSuccess &&
         cudaMemcpyAsync(num_sampled, d_ns, static_cast<size_t>(num_reqs) * 4,
                         cudaMemcpyDeviceToHost, stream) == cudaSuccess &&
         cudaMemcpyAsync(num_rejected, d_nr, static_cast<size_t>(num_reqs) * 4,
                         cudaMemcpyDeviceToHost, stream) == cudaSuccess &&
         cudaStreamSynchronize(stream) == cudaSuccess;
    return ok ? SV_OK : SV_ECUDA;
}

int spec_verify_last_error(spec_verify_ctx *ctx, uint32_t *err_word)
{
    if (!ctx || !err_word) return SV_EINVAL;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
    unsigned w = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&w, ctx->flags + 1, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(ctx->flags + 1, 0, sizeof(unsigned)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return SV_ECUDA;
    *err_word = w;
    return SV_OK;
}

int spec_verify_set_profiling(spec_verify_ctx *ctx, int enable)
{
    if (!ctx) return SV_EINVAL;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
    if (enable && ctx->ring.empty()) {
        ctx->ring.resize(kProfRing);
        for (auto &s : ctx->ring) {
            s.pending = false;
            for (auto &e : s.ev)
                if (cudaEventCreate(&e) != cudaSuccess) return SV_ECUDA;
        }
    }
    ctx->prof = enable != 0;
    return SV_OK;
}

int spec_verify_get_profile(spec_verify_ctx *ctx, double ms[4], int64_t *calls)
{
    if (!ctx || !ms || !calls) return SV_EINVAL;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
    for (auto &s : ctx->ring) prof_collect(ctx, s);
    for (int k = 0; k < kKernels; ++k) {
        ms[k] = ctx->prof_ms[k];
        ctx->prof_ms[k] = 0.0;
    }
    *calls = ctx->prof_done;
    ctx->prof_done = 0;
    return SV_OK;
}

int spec_verify_set_chunks(spec_verify_ctx *ctx, int stats_chunk, int race_chunk)
{
    if (!ctx || stats_chunk < -1 || race_chunk < -1) return SV_EINVAL;
    if (stats_chunk == -1) ctx->stats_chunk = 0;
    else if (stats_chunk) ctx->stats_chunk = round_up8(std::max(stats_chunk, kMinChunk));
    if (race_chunk == -1) ctx->race_chunk = 0;
    else if (race_chunk) ctx->race_chunk = (std::max(race_chunk, kMinChunk) + 15) / 16 * 16;
    return SV_OK;
}

int spec_verify_launches_per_run(void) { return kKernels; }

void spec_verify_free(spec_verify_ctx *ctx)
{
    if (!ctx) return;
    {
        DeviceGuard g(ctx->device);
        cudaDeviceSynchronize();
        free_all(ctx);
    }
    delete ctx;
}

const char *spec_verify_status_string(int status)
{
    switch (status) {
    case SV_OK: return "ok";
    case SV_EINVAL: return "invalid argument";
    case SV_ECAPACITY: return "size above the context capacity";
    case SV_EDTYPE: return "unsupported logits dtype";
    case SV_ECUDA: return "CUDA runtime error";
    case SV_EDEVICE: return "no usable sm_103 device";
    default: return "unknown status";
    }
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Entry point that allocates nothing: the scratch lives in a fixed-size static device array.
// ---------------------------------------------------------------------------------------
namespace {

constexpr int kNoAllocMaxReqs = SV_NOALLOC_MAX_REQS;
constexpr int kNoAllocMaxRows = SV_NOALLOC_MAX_ROWS;
constexpr int kNoAllocMaxVocab = SV_NOALLOC_MAX_VOCAB;
// with the fixed chunk a row spans at most this many CTAs of either kernel
constexpr int kNoAllocMaxSeg = (kNoAllocMaxVocab + kFixedChunk - 1) / kFixedChunk + 1;

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }
constexpr size_t kOffRowInfo = 0;
constexpr size_t kOffRowStat = kOffRowInfo + align256(sizeof(RowInfo) * kNoAllocMaxRows);
constexpr size_t kOffStatPart = kOffRowStat + align256(sizeof(RowStat) * kNoAllocMaxRows);
constexpr size_t kOffReqState =
    kOffStatPart + align256(sizeof(StatPart) * size_t(kNoAllocMaxRows) * kNoAllocMaxSeg);
constexpr size_t kOffRacePart = kOffReqState + align256(sizeof(ReqState) * kNoAllocMaxReqs);
constexpr size_t kOffCounters =
    kOffRacePart + align256(sizeof(RacePart) * size_t(kNoAllocMaxReqs) * kNoAllocMaxSeg);
constexpr size_t kOffFlags =
    kOffCounters + align256(sizeof(unsigned) * counter_words(kNoAllocMaxReqs));
constexpr size_t kNoAllocBytes = kOffFlags + align256(2 * sizeof(unsigned));

// One copy per device that loads this library, kept until the process exits. Every call of
// spec_verify_run_noalloc on a device shares it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_base[kNoAllocMaxDevices] = {};

// Device address of the static scratch on device `dev` (current), looked up once per device
// (the host-side name of the array is not a device address).
int noalloc_base(int dev, void **out)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (!g_noalloc_base[dev]) {
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return SV_ECUDA;
        }
        int a = 0, b = 0, c = 0;
        if (occupancy<uint16_t>(&a, &b, &c) != cudaSuccess || occupancy<float>(&a, &b, &c) != cudaSuccess) {
            cudaGetLastError();
            return SV_ECUDA;
        }
        g_noalloc_base[dev] = p;
    }
    *out = g_noalloc_base[dev];
    return SV_OK;
}

}  // namespace

extern "C" int spec_verify_run_noalloc(const void *logits, int logits_dtype, int vocab_size,
                                       const int32_t *draft_ids, const float *draft_probs,
                                       const int32_t *cu_num_draft, const float *temperature,
                                       const uint8_t *is_greedy, uint64_t seed,
                                       uint32_t req_index_base, int num_reqs, int num_draft_tokens,
                                       int max_spec_len_this_batch, int32_t *sampled,
                                       int32_t *num_sampled, int32_t *num_rejected,
                                       float *opt_row_max, float *opt_row_sumexp,
                                       int32_t *opt_row_argmax, void *cuda_stream)
{
    if (logits_dtype != SV_F32 && logits_dtype != SV_BF16) return SV_EDTYPE;
    if (vocab_size <= 0 || num_reqs < 0 || num_draft_tokens < 0 || max_spec_len_this_batch < 0)
        return SV_EINVAL;
    if (vocab_size > kNoAllocMaxVocab || num_reqs > kNoAllocMaxReqs ||
        static_cast<long long>(num_draft_tokens) + num_reqs > kNoAllocMaxRows ||
        static_cast<long long>(num_draft_tokens) >
            static_cast<long long>(num_reqs) * max_spec_len_this_batch)
        return SV_ECAPACITY;
    if (num_reqs == 0) return SV_OK;
    if (!logits || !cu_num_draft || !temperature || !is_greedy || !sampled || !num_sampled ||
        !num_rejected || (num_draft_tokens > 0 && !draft_ids))
        return SV_EINVAL;
    if (reinterpret_cast<uintptr_t>(logits) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(draft_probs) % 16 != 0)
        return SV_EINVAL;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) {
        cudaGetLastError();
        return SV_EDEVICE;
    }
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess || prop.major != 10 || prop.minor != 3)
        return SV_EDEVICE;
    void *base = nullptr;
    const int rc = noalloc_base(dev, &base);
    if (rc != SV_OK) return rc;
    auto *bytes = static_cast<unsigned char *>(base);

    // A context on the host stack whose scratch pointers are carved from the static array;
    // both kernels use the fixed chunk, so a row never spans more than kNoAllocMaxSeg CTAs.
    spec_verify_ctx view;
    view.device = dev;
    view.max_num_reqs = kNoAllocMaxReqs;
    view.max_spec_len = max_spec_len_this_batch;
    view.V = vocab_size;
    view.dtype = logits_dtype;
    view.has_q = draft_probs != nullptr;
    view.max_rows = kNoAllocMaxRows;
    view.maxseg = kNoAllocMaxSeg;
    view.stats_chunk = kFixedChunk;
    view.race_chunk = kFixedChunk;
    view.rowinfo = reinterpret_cast<RowInfo *>(bytes + kOffRowInfo);
    view.rowstat = reinterpret_cast<RowStat *>(bytes + kOffRowStat);
    view.statpart = reinterpret_cast<StatPart *>(bytes + kOffStatPart);
    view.reqstate = reinterpret_cast<ReqState *>(bytes + kOffReqState);
    view.racepart = reinterpret_cast<RacePart *>(bytes + kOffRacePart);
    view.counters = reinterpret_cast<unsigned *>(bytes + kOffCounters);
    view.flags = reinterpret_cast<unsigned *>(bytes + kOffFlags);
    auto stream = static_cast<cudaStream_t>(cuda_stream);
    if (logits_dtype == SV_BF16)
        return launch_all<uint16_t>(&view, static_cast<const uint16_t *>(logits), draft_ids,
                                    draft_probs, cu_num_draft, temperature, is_greedy, seed,
                                    req_index_base, num_reqs, num_draft_tokens,
                                    max_spec_len_this_batch, sampled, num_sampled, num_rejected,
                                    opt_row_max, opt_row_sumexp, opt_row_argmax, stream);
    return launch_all<float>(&view, static_cast<const float *>(logits), draft_ids, draft_probs,
                             cu_num_draft, temperature, is_greedy, seed, req_index_base, num_reqs,
                             num_draft_tokens, max_spec_len_this_batch, sampled, num_sampled,
                             num_rejected, opt_row_max, opt_row_sumexp, opt_row_argmax, stream);
}
