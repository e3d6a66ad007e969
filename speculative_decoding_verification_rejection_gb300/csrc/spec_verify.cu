// GB300 (sm_103a) implementation of the speculative-decoding verification sampler behind the
// C ABI declared in include/spec_verify.h.
//
// One call = three kernels on the caller's stream, no allocation, no host synchronisation:
//   1. plan   (1 CTA)            validate cu_num_draft, map every logit row to (request, j),
//                                clear the cross-CTA counters.
//   2. stats  (rows x splits)    stream the logits once: per row m = max x, S = sum exp(x - m),
//                                raw argmax ([spec-in-vllm] 7.4 block stats); the last CTA of a
//                                row combines the splits and runs the row's acceptance test
//                                ([spec-notes] 8.3 / NO_DRAFT_PROBS answer code).
//   3. race   (requests x splits) per request: scan the acceptance flags for the first
//                                rejection j* ([MTP-eagle] _rejection_sample_kernel), race the
//                                one row that is emitted (residual max(0, p - q), p without the
//                                rejected draft, or p for the bonus / non-speculative draw,
//                                [spec-notes] residual and NO_DRAFT_PROBS answers, [spec-in-vllm]
//                                7.3), and the last CTA writes sampled / num_sampled /
//                                num_rejected.
// Only the emitted row of a request is raced: a residual that is never emitted cannot change
// any output, so its logits and q row are never read.
#include <cuda_runtime.h>

#include <climits>
#include <cstddef>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "spec_verify.h"
#include "sv_device.cuh"

namespace {

constexpr int kThreads = 256;
constexpr int kPlanThreads = 1024;
constexpr int kMinChunk = 2048;        // smallest elements per CTA (sizes the partial buffers)
constexpr int kDefaultStatsChunk = 16384;
constexpr int kDefaultRaceChunk = 8192;
constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kInf = __builtin_huge_valf();

enum : int32_t { kFlagGreedy = 1, kFlagBonus = 2 };

struct __align__(16) RowInfo {
    int32_t req;   // request index within the call
    int32_t j;     // position, K = bonus
    int32_t flags; // kFlagGreedy | kFlagBonus
    float invT;    // 1 / T (1 for greedy rows)
};

struct __align__(16) ReqInfo {
    int32_t q0;    // cu_num_draft[i]
    int32_t K;     // draft length
    int32_t flags;
    float invT;
};

struct __align__(16) RowStat {
    float m;       // max_v x_v
    float S;       // sum_v exp(x_v - m)
    int32_t amax;  // raw-logit argmax, lowest index
    int32_t acc;   // acceptance of the row's draft (bonus rows: 1)
};

struct __align__(16) StatPart {
    float L;       // max raw logit of the split
    float s;       // sum of 2^((l - L) c) over the split
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
// 1. plan
// ---------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kPlanThreads)
sv_plan_kernel(const int32_t *__restrict__ cu, const float *__restrict__ temperature,
               const uint8_t *__restrict__ is_greedy, int num_reqs, int num_draft_tokens,
               int kmax, RowInfo *__restrict__ rowinfo, ReqInfo *__restrict__ reqinfo,
               unsigned *__restrict__ row_counter, int num_rows,
               unsigned *__restrict__ req_counter, unsigned *__restrict__ flags)
{
    __shared__ int bad;
    if (threadIdx.x == 0) bad = (cu[0] != 0) || (cu[num_reqs] != num_draft_tokens);
    __syncthreads();
    for (int r = threadIdx.x; r < num_rows; r += blockDim.x) row_counter[r] = 0u;
    for (int i = threadIdx.x; i < num_reqs; i += blockDim.x) {
        req_counter[i] = 0u;
        const int lo = cu[i], hi = cu[i + 1];
        const int K = hi - lo;
        if (K < 0 || K > kmax || lo < 0 || hi > num_draft_tokens) {
            bad = 1;
            continue;
        }
        const float T = temperature[i];
        const bool greedy = is_greedy[i] != 0 || !(T > 0.0f);
        const float invT = greedy ? 1.0f : __frcp_rn(T);
        const int32_t gf = greedy ? kFlagGreedy : 0;
        reqinfo[i] = ReqInfo{lo, K, gf, invT};
        for (int j = 0; j <= K; ++j)
            rowinfo[lo + i + j] = RowInfo{i, j, gf | (j == K ? kFlagBonus : 0), invT};
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        flags[0] = bad ? 1u : 0u;
        if (bad) atomicOr(&flags[1], SV_ERR_BATCH);
    }
}

// ---------------------------------------------------------------------------------------
// 2. row statistics + acceptance test
// ---------------------------------------------------------------------------------------
struct OnlineMax {
    float L = -kInf;   // running max of raw logits
    float s = 0.0f;    // running sum of 2^((l - L) c)
    int idx = INT_MAX; // lowest index of L
    float Lc = -kInf;  // L * c
};

// Fold a group of n raw logits starting at index e0 (indices increase within a thread).
template <int N>
__device__ __forceinline__ void fold(OnlineMax &st, const float (&l)[N], int e0, float c)
{
    float mx = l[0];
#pragma unroll
    for (int k = 1; k < N; ++k) mx = fmaxf(mx, l[k]);
    if (mx > st.L) {
        int kk = 0;
#pragma unroll
        for (int k = N - 1; k >= 0; --k)
            if (l[k] == mx) kk = k;
        st.s = st.s == 0.0f ? 0.0f : st.s * sv::ex2_approx((st.L - mx) * c);
        st.L = mx;
        st.Lc = mx * c;
        st.idx = e0 + kk;
    }
    if (st.L > -kInf) {
#pragma unroll
        for (int k = 0; k < N; ++k) st.s += sv::ex2_approx(fmaf(l[k], c, -st.Lc));
    }
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

template <typename T>
__global__ void __launch_bounds__(kThreads)
sv_stats_kernel(const T *__restrict__ logits, int V, int chunk, int splits,
                const RowInfo *__restrict__ rowinfo, RowStat *__restrict__ rowstat,
                StatPart *__restrict__ part, unsigned *__restrict__ row_counter,
                const int32_t *__restrict__ draft_ids, const float *__restrict__ q, uint64_t seed,
                uint32_t req_base, float *__restrict__ opt_max, float *__restrict__ opt_sum,
                int32_t *__restrict__ opt_amax, const unsigned *__restrict__ flags)
{
    if (flags[0]) return;
    const int row = blockIdx.x / splits;
    const int sp = blockIdx.x - row * splits;
    const RowInfo ri = rowinfo[row];
    const float c = ri.invT * kLog2e;
    const T *rp = logits + static_cast<size_t>(row) * static_cast<size_t>(V);
    const int begin = sp * chunk;
    const int end = min(V, begin + chunk);

    constexpr int kVec = 16 / sizeof(T);  // elements per 16-byte load
    const uintptr_t addr = reinterpret_cast<uintptr_t>(rp + begin);
    const int head = static_cast<int>(((16u - (addr & 15u)) & 15u) / sizeof(T));
    const int a0 = min(end, begin + head);
    const int nvec = (end - a0) / kVec;
    const int a1 = a0 + nvec * kVec;

    OnlineMax st;
    for (int e = begin + threadIdx.x; e < a0; e += kThreads) {
        const float l[1] = {Elem<T>::at(rp, e)};
        fold<1>(st, l, e, c);
    }
    const char *vbase = reinterpret_cast<const char *>(rp + a0);
    constexpr int kUnroll = 4;
    for (int u0 = threadIdx.x; u0 < nvec; u0 += kThreads * kUnroll) {
        uint4 w[kUnroll];
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int u = u0 + k * kThreads;
            w[k] = u < nvec ? ldg_v4(vbase + static_cast<size_t>(u) * 16) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < kUnroll; ++k) {
            const int u = u0 + k * kThreads;
            if (u >= nvec) break;
            const int e0 = a0 + u * kVec;
            if constexpr (sizeof(T) == 2) {
                const float l[8] = {__uint_as_float(w[k].x << 16), __uint_as_float(w[k].x & 0xFFFF0000u),
                                    __uint_as_float(w[k].y << 16), __uint_as_float(w[k].y & 0xFFFF0000u),
                                    __uint_as_float(w[k].z << 16), __uint_as_float(w[k].z & 0xFFFF0000u),
                                    __uint_as_float(w[k].w << 16), __uint_as_float(w[k].w & 0xFFFF0000u)};
                fold<8>(st, l, e0, c);
            } else {
                const float l[4] = {__uint_as_float(w[k].x), __uint_as_float(w[k].y),
                                    __uint_as_float(w[k].z), __uint_as_float(w[k].w)};
                fold<4>(st, l, e0, c);
            }
        }
    }
    for (int e = a1 + threadIdx.x; e < end; e += kThreads) {
        const float l[1] = {Elem<T>::at(rp, e)};
        fold<1>(st, l, e, c);
    }

    float L = st.L, s = st.s;
    int idx = st.idx;
    block_reduce_stat(L, s, idx, c);

    __shared__ int s_last;
    if (splits > 1) {
        if (threadIdx.x == 0) {
            part[static_cast<size_t>(row) * splits + sp] = StatPart{L, s, idx, 0};
            __threadfence();
            const unsigned ticket = atomicAdd(&row_counter[row], 1u);
            s_last = ticket == static_cast<unsigned>(splits - 1);
        }
        __syncthreads();
        if (!s_last) return;
        // Last CTA of the row: combine the splits in a fixed order (deterministic).
        __threadfence();
        if (threadIdx.x < 32) {
            const int lane = threadIdx.x;
            float Lw = -kInf, sw = 0.0f;
            int iw = INT_MAX;
            for (int k = lane; k < splits; k += 32) {
                const float4 raw = __ldcg(reinterpret_cast<const float4 *>(part) +
                                          static_cast<size_t>(row) * splits + k);
                combine_stat(Lw, sw, iw, raw.x, raw.y, __float_as_int(raw.z), c);
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float L2 = __shfl_xor_sync(0xFFFFFFFFu, Lw, o);
                const float s2 = __shfl_xor_sync(0xFFFFFFFFu, sw, o);
                const int i2 = __shfl_xor_sync(0xFFFFFFFFu, iw, o);
                combine_stat(Lw, sw, iw, L2, s2, i2, c);
            }
            L = Lw;
            s = sw;
            idx = iw;
            if (lane == 0) row_counter[row] = 0u;
        }
    }
    if (threadIdx.x != 0) return;

    // Row finaliser (one thread).
    const float m = __fmul_rn(L, ri.invT);  // = max_v fl(l_v / T): rounding is monotone
    const int amax = idx == INT_MAX ? 0 : idx;
    int acc = 1;
    if (!(ri.flags & kFlagBonus)) {
        const int qrow = row - ri.req;  // cu_num_draft[i] + j
        const int d = draft_ids[qrow];
        if (ri.flags & kFlagGreedy) {
            acc = d == amax;
        } else if (d < 0 || d >= V) {
            acc = 0;
        } else {
            const float x_d = __fmul_rn(Elem<T>::at(rp, d), ri.invT);
            const float t_d = sv::exp_f32(__fsub_rn(x_d, m));
            const float p_d = __fdiv_rn(t_d, s);
            const float q_d = q ? __ldg(q + static_cast<size_t>(qrow) * V + d) : 1.0f;
            const sv::Philox4 r = sv::philox4x32_10(0u, static_cast<uint32_t>(ri.j),
                                                    req_base + static_cast<uint32_t>(ri.req),
                                                    sv::kTagAccept, static_cast<uint32_t>(seed),
                                                    static_cast<uint32_t>(seed >> 32));
            const float u = sv::uniform_from_word(r.x);
            acc = (q_d > 0.0f) && (__fdiv_rn(p_d, q_d) >= u);
        }
    }
    rowstat[row] = RowStat{m, s, amax, acc};
    if (opt_max) opt_max[row] = m;
    if (opt_sum) opt_sum[row] = s;
    if (opt_amax) opt_amax[row] = amax;
}

// ---------------------------------------------------------------------------------------
// 3. race + scan + emit
// ---------------------------------------------------------------------------------------
struct RaceState {
    float kb = -kInf;  // best key so far
    int ib = -1;       // its index (-1: none yet)
    // screening constants derived from kb (see refresh)
    float pre_x;       // p-race: skip a group whose max x is below this
    float kbl;         // p-race: (kb - delta) * log2 e
    float pre_rr;      // residual: skip a group whose rr upper bounds are all below this
    float ekb;         // residual: >= exp(delta - kb)
};

constexpr float kSafe = 1.0f + 0x1p-10f;  // covers MUFU and argument rounding errors

__device__ __forceinline__ void refresh(RaceState &st)
{
    if (st.ib < 0) {
        st.pre_x = -kInf;
        st.kbl = -kInf;
        st.pre_rr = -kInf;
        st.ekb = kInf;
        return;
    }
    const float delta = 1e-3f + 1e-5f * fabsf(st.kb);
    st.pre_x = st.kb - (sv::kGumbelMax + delta);
    st.kbl = (st.kb - delta) * kLog2e;
    st.pre_rr = sv::ex2_approx((st.kb - sv::kGumbelMax - delta) * kLog2e) * (1.0f - 0x1p-9f);
    st.ekb = sv::ex2_approx((delta - st.kb) * kLog2e) * kSafe;
}

__device__ __forceinline__ bool race_better(float ka, int ia, float kb, int ib)
{
    // is (ka, ia) better than (kb, ib)? larger key, then lower index; -1 = no candidate
    if (ia < 0) return false;
    if (ib < 0) return true;
    return ka > kb || (ka == kb && ia < ib);
}

// Offer element v: x = logit / T, U its race uniform. Returns after the full key only if the
// conservative screen could not rule it out.
template <bool kResidual>
__device__ __forceinline__ void race_offer(RaceState &st, int v, float x, float qv, float U,
                                           float m, float S, float rr_up)
{
    const float om = 1.0f - U;  // exact
    if constexpr (kResidual) {
        if (!(rr_up > 0.0f)) return;
        // key < kb is certain if -log U >= 1 - U > rr * exp(delta - kb)
        if (om > rr_up * st.ekb) return;
        const float t = sv::exp_f32(__fsub_rn(x, m));
        const float rr = __fmaf_rn(-S, qv, t);
        if (!(rr > 0.0f)) return;
        const float E = -sv::log_f32(U);
        const float key = __fsub_rn(sv::log_f32(rr), sv::log_f32(E));
        if (st.ib < 0 || key > st.kb) {
            st.kb = key;
            st.ib = v;
            refresh(st);
        }
    } else {
        if (om > sv::ex2_approx(fmaf(x, kLog2e, -st.kbl)) * kSafe) return;
        const float E = -sv::log_f32(U);
        const float key = __fsub_rn(x, sv::log_f32(E));
        if (st.ib < 0 || key > st.kb) {
            st.kb = key;
            st.ib = v;
            refresh(st);
        }
    }
}

// Race over [b, e) of one row (b a multiple of 4). Groups of 4 consecutive tokens share one
// Philox call (counter word 0 = v >> 2).
template <typename T, bool kResidual>
__device__ __forceinline__ void race_span(RaceState &st, const T *__restrict__ rp,
                                          const float *__restrict__ qrow, int b, int e,
                                          float invT, float m, float S, int exclude, uint32_t j,
                                          uint32_t ireq, uint32_t k0, uint32_t k1, bool aligned)
{
    for (int g0 = b + 4 * static_cast<int>(threadIdx.x); g0 < e; g0 += 4 * kThreads) {
        const int n = min(4, e - g0);
        float x[4], qv[4] = {0.f, 0.f, 0.f, 0.f};
        if (aligned && n == 4) {
            if constexpr (sizeof(T) == 2) {
                const uint2 w = __ldg(reinterpret_cast<const uint2 *>(rp + g0));
                x[0] = __uint_as_float(w.x << 16);
                x[1] = __uint_as_float(w.x & 0xFFFF0000u);
                x[2] = __uint_as_float(w.y << 16);
                x[3] = __uint_as_float(w.y & 0xFFFF0000u);
            } else {
                const float4 w = __ldg(reinterpret_cast<const float4 *>(rp + g0));
                x[0] = w.x; x[1] = w.y; x[2] = w.z; x[3] = w.w;
            }
            if constexpr (kResidual) {
                const float4 w = __ldg(reinterpret_cast<const float4 *>(qrow + g0));
                qv[0] = w.x; qv[1] = w.y; qv[2] = w.z; qv[3] = w.w;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                x[k] = k < n ? Elem<T>::at(rp, g0 + k) : -kInf;
                if constexpr (kResidual) qv[k] = k < n ? __ldg(qrow + g0 + k) : 0.0f;
            }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) x[k] = __fmul_rn(x[k], invT);

        float rr_up[4] = {0.f, 0.f, 0.f, 0.f};
        if constexpr (kResidual) {
            float mx = -kInf;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float t_up = sv::ex2_approx((x[k] - m) * kLog2e) * kSafe;
                rr_up[k] = k < n ? fmaf(-S, qv[k], t_up) : -kInf;
                mx = fmaxf(mx, rr_up[k]);
            }
            if (!(mx > 0.0f) || mx < st.pre_rr) continue;
        } else {
            const float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
            if (mx < st.pre_x) continue;
        }
        const sv::Philox4 r = sv::philox4x32_10(static_cast<uint32_t>(g0) >> 2, j, ireq,
                                                sv::kTagRace, k0, k1);
        const uint32_t words[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int v = g0 + k;
            if (k >= n || v == exclude) continue;
            race_offer<kResidual>(st, v, x[k], qv[k], sv::uniform_from_word(words[k]), m, S,
                                  rr_up[k]);
        }
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

template <typename T>
__device__ void race_row(float &kb, int &ib, const T *rp, const float *qrow, int b, int e,
                         float invT, float m, float S, int exclude, uint32_t j, uint32_t ireq,
                         uint64_t seed, bool aligned)
{
    RaceState st;
    refresh(st);
    const uint32_t k0 = static_cast<uint32_t>(seed), k1 = static_cast<uint32_t>(seed >> 32);
    if (qrow)
        race_span<T, true>(st, rp, qrow, b, e, invT, m, S, exclude, j, ireq, k0, k1, aligned);
    else
        race_span<T, false>(st, rp, qrow, b, e, invT, m, S, exclude, j, ireq, k0, k1, aligned);
    kb = st.kb;
    ib = st.ib;
    block_reduce_race(kb, ib);
}

__device__ __forceinline__ void emit(int i, int jstar, int K, int q0, int token,
                                     const int32_t *__restrict__ draft_ids,
                                     int32_t *__restrict__ sampled, int stride,
                                     int32_t *__restrict__ num_sampled,
                                     int32_t *__restrict__ num_rejected)
{
    int32_t *out = sampled + static_cast<size_t>(i) * stride;
    for (int s = threadIdx.x; s < stride; s += blockDim.x)
        out[s] = s < jstar ? draft_ids[q0 + s] : (s == jstar ? token : -1);
    if (threadIdx.x == 0) {
        num_sampled[i] = jstar + 1;
        num_rejected[i] = jstar < 0 ? 0 : K - jstar;
    }
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
sv_race_kernel(const T *__restrict__ logits, int V, int chunk, int splits,
               const ReqInfo *__restrict__ reqinfo, const RowStat *__restrict__ rowstat,
               const int32_t *__restrict__ draft_ids, const float *__restrict__ q, uint64_t seed,
               uint32_t req_base, RacePart *__restrict__ part, unsigned *__restrict__ req_counter,
               int32_t *__restrict__ sampled, int stride, int32_t *__restrict__ num_sampled,
               int32_t *__restrict__ num_rejected, const unsigned *__restrict__ flags,
               bool aligned)
{
    const int i = blockIdx.x / splits;
    const int sp = blockIdx.x - i * splits;
    if (flags[0]) {
        if (sp == 0) emit(i, -1, 0, 0, -1, draft_ids, sampled, stride, num_sampled, num_rejected);
        return;
    }
    const ReqInfo rq = reqinfo[i];
    const int row0 = rq.q0 + i;

    __shared__ int s_jstar;
    if (threadIdx.x < 32) {
        const int lane = threadIdx.x;
        int js = rq.K;
        for (int jb = 0; jb < rq.K; jb += 32) {
            const int j = jb + lane;
            const bool rej = j < rq.K && rowstat[row0 + j].acc == 0;
            const unsigned msk = __ballot_sync(0xFFFFFFFFu, rej);
            if (msk) {
                js = jb + __ffs(msk) - 1;
                break;
            }
        }
        if (lane == 0) s_jstar = js;
    }
    __syncthreads();
    const int js = s_jstar;

    if (rq.flags & kFlagGreedy) {
        // [spec-notes] 8.3 greedy: the target argmax at the mismatch, or of the bonus row
        if (sp == 0)
            emit(i, js, rq.K, rq.q0, rowstat[row0 + js].amax, draft_ids, sampled, stride,
                 num_sampled, num_rejected);
        return;
    }

    const RowStat rs = rowstat[row0 + js];
    const T *rp = logits + static_cast<size_t>(row0 + js) * static_cast<size_t>(V);
    const bool rejected = js < rq.K;
    const float *qrow = (rejected && q) ? q + static_cast<size_t>(rq.q0 + js) * V : nullptr;
    const int exclude = (rejected && !q) ? draft_ids[rq.q0 + js] : -1;
    const uint32_t ireq = req_base + static_cast<uint32_t>(i);
    const int b = sp * chunk;
    const int e = min(V, b + chunk);

    float kb;
    int ib;
    race_row<T>(kb, ib, rp, qrow, b, e, rq.invT, rs.m, rs.S, exclude, static_cast<uint32_t>(js),
                ireq, seed, aligned);

    __shared__ int s_last;
    __shared__ int s_token;
    if (splits > 1) {
        if (threadIdx.x == 0) {
            part[static_cast<size_t>(i) * splits + sp] = RacePart{kb, ib};
            __threadfence();
            const unsigned ticket = atomicAdd(&req_counter[i], 1u);
            s_last = ticket == static_cast<unsigned>(splits - 1);
        }
        __syncthreads();
        if (!s_last) return;
        __threadfence();
        if (threadIdx.x < 32) {
            float kw = -kInf;
            int iw = -1;
            for (int k = threadIdx.x; k < splits; k += 32) {
                const float2 raw = __ldcg(reinterpret_cast<const float2 *>(part) +
                                          static_cast<size_t>(i) * splits + k);
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
                req_counter[i] = 0u;
            }
        }
    }
    if (threadIdx.x == 0) s_token = ib;
    __syncthreads();
    int token = s_token;
    if (token < 0) {
        // Nothing left after rounding (residual with p <= q everywhere, or V == 1 with the only
        // token excluded): draw from p itself so the output stays a target-side draw.
        race_row<T>(kb, ib, rp, nullptr, 0, V, rq.invT, rs.m, rs.S, -1,
                    static_cast<uint32_t>(js), ireq, seed, aligned);
        if (threadIdx.x == 0) s_token = ib;
        __syncthreads();
        token = s_token;
    }
    emit(i, js, rq.K, rq.q0, token, draft_ids, sampled, stride, num_sampled, num_rejected);
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
constexpr int kProfRing = 512;

struct ProfSlot {
    cudaEvent_t ev[4];
    bool pending;
};

int round_up8(int x) { return (x + 7) / 8 * 8; }
int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace

struct spec_verify_ctx {
    int device = 0;
    int max_num_reqs = 0, max_spec_len = 0, V = 0, dtype = SV_F32, has_q = 0;
    int max_rows = 0, max_splits = 0;
    int stats_chunk = kDefaultStatsChunk, race_chunk = kDefaultRaceChunk;
    RowInfo *rowinfo = nullptr;
    ReqInfo *reqinfo = nullptr;
    RowStat *rowstat = nullptr;
    StatPart *statpart = nullptr;
    RacePart *racepart = nullptr;
    unsigned *counters = nullptr;  // [max_rows] row counters, [max_num_reqs] request counters
    unsigned *flags = nullptr;     // [0] per-call batch-invalid, [1] sticky error word
    // host-buffer staging
    void *io_logits = nullptr;
    float *io_q = nullptr;
    int32_t *io_small = nullptr;   // ids | cu | sampled | num_sampled | num_rejected
    float *io_temp = nullptr;
    uint8_t *io_greedy = nullptr;
    // profiling
    bool prof = false;
    std::vector<ProfSlot> ring;
    int64_t prof_calls = 0, prof_done = 0;
    double prof_ms[3] = {0, 0, 0};
};

namespace {

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
    cudaEventSynchronize(s.ev[3]);
    for (int k = 0; k < 3; ++k) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, s.ev[k], s.ev[k + 1]) == cudaSuccess) ctx->prof_ms[k] += ms;
    }
    s.pending = false;
    ctx->prof_done++;
}

void free_all(spec_verify_ctx *ctx)
{
    cudaFree(ctx->rowinfo);
    cudaFree(ctx->reqinfo);
    cudaFree(ctx->rowstat);
    cudaFree(ctx->statpart);
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

template <typename T>
int launch_all(spec_verify_ctx *ctx, const T *logits, const int32_t *draft_ids, const float *q,
               const int32_t *cu, const float *temperature, const uint8_t *is_greedy,
               uint64_t seed, uint32_t base, int num_reqs, int nd, int kmax, int32_t *sampled,
               int32_t *num_sampled, int32_t *num_rejected, float *opt_max, float *opt_sum,
               int32_t *opt_amax, cudaStream_t stream)
{
    const int V = ctx->V;
    const int rows = nd + num_reqs;
    const int chunk1 = min(round_up8(ctx->stats_chunk), round_up8(V));
    const int splits1 = ceil_div(V, chunk1);
    const int chunk2 = min(round_up8(ctx->race_chunk), round_up8(V));
    const int splits2 = ceil_div(V, chunk2);
    // Groups of 4 tokens start on 8-byte (bf16) / 16-byte (fp32, q) boundaries when V % 4 == 0
    // (base pointers are checked to be 16-byte aligned): the race can use vector loads.
    const bool aligned = V % 4 == 0;
    unsigned *row_counter = ctx->counters;
    unsigned *req_counter = ctx->counters + ctx->max_rows;

    ProfSlot *slot = nullptr;
    if (ctx->prof) {
        slot = &ctx->ring[static_cast<size_t>(ctx->prof_calls % kProfRing)];
        prof_collect(ctx, *slot);
        cudaEventRecord(slot->ev[0], stream);
    }
    sv_plan_kernel<<<1, kPlanThreads, 0, stream>>>(cu, temperature, is_greedy, num_reqs, nd, kmax,
                                                   ctx->rowinfo, ctx->reqinfo, row_counter, rows,
                                                   req_counter, ctx->flags);
    if (slot) cudaEventRecord(slot->ev[1], stream);
    sv_stats_kernel<T><<<rows * splits1, kThreads, 0, stream>>>(
        logits, V, chunk1, splits1, ctx->rowinfo, ctx->rowstat, ctx->statpart, row_counter,
        draft_ids, q, seed, base, opt_max, opt_sum, opt_amax, ctx->flags);
    if (slot) cudaEventRecord(slot->ev[2], stream);
    sv_race_kernel<T><<<num_reqs * splits2, kThreads, 0, stream>>>(
        logits, V, chunk2, splits2, ctx->reqinfo, ctx->rowstat, draft_ids, q, seed, base,
        ctx->racepart, req_counter, sampled, kmax + 1, num_sampled, num_rejected, ctx->flags,
        aligned);
    if (slot) {
        cudaEventRecord(slot->ev[3], stream);
        slot->pending = true;
        ctx->prof_calls++;
    }
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
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
    if (rows > INT_MAX / 8 || static_cast<long long>(max_num_reqs) * ceil_div(vocab_size, kMinChunk) > INT_MAX / 2)
        return SV_ECAPACITY;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return SV_EDEVICE;
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
    ctx->max_splits = ceil_div(vocab_size, kMinChunk);
    const size_t R = static_cast<size_t>(rows), N = static_cast<size_t>(max_num_reqs);
    const size_t P = static_cast<size_t>(ctx->max_splits);
    bool ok = cudaMalloc(&ctx->rowinfo, R * sizeof(RowInfo)) == cudaSuccess &&
              cudaMalloc(&ctx->reqinfo, N * sizeof(ReqInfo)) == cudaSuccess &&
              cudaMalloc(&ctx->rowstat, R * sizeof(RowStat)) == cudaSuccess &&
              cudaMalloc(&ctx->statpart, R * P * sizeof(StatPart)) == cudaSuccess &&
              cudaMalloc(&ctx->racepart, N * P * sizeof(RacePart)) == cudaSuccess &&
              cudaMalloc(&ctx->counters, (R + N) * sizeof(unsigned)) == cudaSuccess &&
              cudaMalloc(&ctx->flags, 2 * sizeof(unsigned)) == cudaSuccess;
    ok = ok && cudaMemset(ctx->counters, 0, (R + N) * sizeof(unsigned)) == cudaSuccess &&
         cudaMemset(ctx->flags, 0, 2 * sizeof(unsigned)) == cudaSuccess &&
         cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
        free_all(ctx);
        delete ctx;
        cudaGetLastError();
        return SV_ECUDA;
    }
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
    if (num_reqs < 0 || num_draft_tokens < 0 || max_spec_len_this_batch < 0) return SV_EINVAL;
    if (num_reqs > ctx->max_num_reqs || max_spec_len_this_batch > ctx->max_spec_len ||
        static_cast<long long>(num_draft_tokens) >
            static_cast<long long>(num_reqs) * max_spec_len_this_batch)
        return SV_ECAPACITY;
    if (num_reqs == 0) return SV_OK;
    if (!logits || !cu_num_draft || !temperature || !is_greedy || !sampled || !num_sampled ||
        !num_rejected || (num_draft_tokens > 0 && !draft_ids))
        return SV_EINVAL;
    if (draft_probs && !ctx->has_q) return SV_EINVAL;
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
        ctx->io_logits = ctx->io_q = nullptr;
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
    if (num_reqs < 0 || num_draft_tokens < 0 || max_spec_len_this_batch < 0) return SV_EINVAL;
    if (num_reqs > ctx->max_num_reqs || max_spec_len_this_batch > ctx->max_spec_len ||
        static_cast<long long>(num_draft_tokens) >
            static_cast<long long>(num_reqs) * max_spec_len_this_batch)
        return SV_ECAPACITY;
    if (num_reqs == 0) return SV_OK;
    if (!logits || !cu_num_draft || !temperature || !is_greedy || !sampled || !num_sampled ||
        !num_rejected || (num_draft_tokens > 0 && !draft_ids))
        return SV_EINVAL;
    if (draft_probs && !ctx->has_q) return SV_EINVAL;
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
    int rc = spec_verify_run(ctx, ctx->io_logits, d_ids, draft_probs ? ctx->io_q : nullptr, d_cu,
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

int spec_verify_get_profile(spec_verify_ctx *ctx, double ms[3], int64_t *calls)
{
    if (!ctx || !ms || !calls) return SV_EINVAL;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
    for (auto &s : ctx->ring) prof_collect(ctx, s);
    for (int k = 0; k < 3; ++k) {
        ms[k] = ctx->prof_ms[k];
        ctx->prof_ms[k] = 0.0;
    }
    *calls = ctx->prof_done;
    ctx->prof_done = 0;
    return SV_OK;
}

int spec_verify_set_chunks(spec_verify_ctx *ctx, int stats_chunk, int race_chunk)
{
    if (!ctx || stats_chunk < 0 || race_chunk < 0) return SV_EINVAL;
    if (stats_chunk) ctx->stats_chunk = round_up8(stats_chunk < kMinChunk ? kMinChunk : stats_chunk);
    if (race_chunk) ctx->race_chunk = round_up8(race_chunk < kMinChunk ? kMinChunk : race_chunk);
    return SV_OK;
}

int spec_verify_launches_per_run(void) { return 3; }

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
#include <mutex>

namespace {

constexpr int kNoAllocMaxReqs = SV_NOALLOC_MAX_REQS;
constexpr int kNoAllocMaxRows = SV_NOALLOC_MAX_ROWS;
constexpr int kNoAllocMaxVocab = SV_NOALLOC_MAX_VOCAB;
constexpr int kNoAllocSplits1 = (kNoAllocMaxVocab + kDefaultStatsChunk - 1) / kDefaultStatsChunk;
constexpr int kNoAllocSplits2 = (kNoAllocMaxVocab + kDefaultRaceChunk - 1) / kDefaultRaceChunk;

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }
constexpr size_t kOffRowInfo = 0;
constexpr size_t kOffRowStat = kOffRowInfo + align256(sizeof(RowInfo) * kNoAllocMaxRows);
constexpr size_t kOffStatPart = kOffRowStat + align256(sizeof(RowStat) * kNoAllocMaxRows);
constexpr size_t kOffCounters =
    kOffStatPart + align256(sizeof(StatPart) * size_t(kNoAllocMaxRows) * kNoAllocSplits1);
constexpr size_t kOffFlags =
    kOffCounters + align256(sizeof(unsigned) * size_t(kNoAllocMaxRows + kNoAllocMaxReqs));
constexpr size_t kOffReqInfo = kOffFlags + align256(2 * sizeof(unsigned));
constexpr size_t kOffRacePart = kOffReqInfo + align256(sizeof(ReqInfo) * kNoAllocMaxReqs);
constexpr size_t kNoAllocBytes =
    kOffRacePart + align256(sizeof(RacePart) * size_t(kNoAllocMaxReqs) * kNoAllocSplits2);

// One copy per device that loads this library, kept until the process exits. Every call of
// spec_verify_run_noalloc on a device shares it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_base[kNoAllocMaxDevices] = {};

// Device address of the static scratch on the current device, looked up once per device
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

    // A context on the host stack whose scratch pointers are carved from the static array.
    spec_verify_ctx view;
    view.device = dev;
    view.max_num_reqs = kNoAllocMaxReqs;
    view.max_spec_len = max_spec_len_this_batch;
    view.V = vocab_size;
    view.dtype = logits_dtype;
    view.has_q = draft_probs != nullptr;
    view.max_rows = kNoAllocMaxRows;
    view.max_splits = kNoAllocSplits2;
    view.rowinfo = reinterpret_cast<RowInfo *>(bytes + kOffRowInfo);
    view.rowstat = reinterpret_cast<RowStat *>(bytes + kOffRowStat);
    view.statpart = reinterpret_cast<StatPart *>(bytes + kOffStatPart);
    view.counters = reinterpret_cast<unsigned *>(bytes + kOffCounters);
    view.flags = reinterpret_cast<unsigned *>(bytes + kOffFlags);
    view.reqinfo = reinterpret_cast<ReqInfo *>(bytes + kOffReqInfo);
    view.racepart = reinterpret_cast<RacePart *>(bytes + kOffRacePart);
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
