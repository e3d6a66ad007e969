// GB300 (sm_103a) implementation of the speculative-decoding verification sampler behind the
// C ABI declared in include/spec_verify.h.
//
// One call = two kernels on the caller's stream, no allocation, no host synchronisation:
//   1. stats  (whole waves)      stream every logit once, the flattened [rows x V] array split
//                                evenly over the CTAs; each CTA looks its rows' requests up in
//                                cu_num_draft (for the temperature) and writes one partial
//                                (max, sum of exp, argmax) per row segment ([spec-in-vllm] 7.4
//                                block stats).
//   2. verify (CTA per request)  validate cu_num_draft; combine each row's partials into
//                                m = max x, S = sum exp(x - m) and the raw argmax; test every
//                                draft ([spec-notes] 8.3 and the NO_DRAFT_PROBS answer code);
//                                find the first rejection j* ([MTP-eagle]
//                                _rejection_sample_kernel); emit the argmax there for a greedy
//                                request, or draw the token at j* for a sampling request by the
//                                exponential race over the residual max(0, p - q), over p without
//                                the rejected draft, or over p for the bonus draw ([spec-notes]
//                                residual and NO_DRAFT_PROBS answers, [spec-in-vllm] 7.3).
//
// The race is a best-first search, not a scan. Keys are w_v / E_v with w_v = exp(x_v - m) (a
// race over p) or the residual weight (at most exp(x_v - m)). A row's race clocks come in groups
// of 64 tokens whose head Philox call gives the group's smallest clock E_g, so no key in group g
// exceeds exp(max_{v in g} x_v - m) / E_g. The verify CTA takes the largest logit of every
// 64-element line of the raced row (written by the statistics kernel), bounds every group with
// one Philox call, evaluates first the groups with the best bounds and then only the groups whose
// bound still reaches the best key found -- a few dozen of the V / 64 groups on typical rows. Only
// exact keys decide, so the winner is the argmax over all tokens, as a full scan would find it;
// only the line maxima of the raced row and the logits and q entries of evaluated groups are read.
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstddef>
#include <cstdint>
#include <cstdlib>
#include <mutex>
#include <new>
#include <vector>

#include "spec_verify.h"
#include "sv_device.cuh"

namespace {

constexpr int kThreads = 256;       // both kernels
constexpr int kWarps = kThreads / 32;
constexpr int kMinChunk = 2048;     // smallest elements per statistics CTA (bounds the partials)
constexpr int kChunkAlign = 512;    // statistics chunks: whole 16-byte spans of the line array
constexpr int kMaxChunk = 1 << 19;  // largest: its line maxima fit in 32 KB of shared memory
constexpr int kFixedChunk = 32768;  // statistics chunk of the static-scratch entry point
constexpr int kGroup = 64;          // tokens per race-clock group = elements per line
constexpr float kLog2e = 0x1.715476p+0f;
constexpr float kInf = __builtin_huge_valf();

struct __align__(16) StatPart {
    float L;       // max raw logit of the segment
    float s;       // sum of 2^((l - L) c) over the segment
    int32_t idx;   // where L first occurs, as a candidate (see argmax_candidate)
    int32_t pad;
};

// A partial's first occurrence of its maximum, ordered like the index it stands for: 2 e for
// element e of the row, 2 a + 1 for the 64-byte pair starting at element a (its lowest element
// equal to the maximum is the one; the reader resolves it, only when it needs the index), and
// INT_MAX for none. Elements and pairs of one row never overlap, so the smallest candidate among
// partials tied at the row maximum holds the row's first occurrence. Indices stay below 2^30.
__device__ __forceinline__ int argmax_candidate(int e, bool pair) { return (e << 1) | (pair ? 1 : 0); }

// ---------------------------------------------------------------------------------------
// checked global memory access (debug builds)
// ---------------------------------------------------------------------------------------
// Built with -DSV_DEBUG_BOUNDS, the library checks every global load and store of its kernels
// against the arrays of the current call (their address ranges, registered by the host before
// the launches): an access outside all of them is skipped (a load gives 0) and sets
// SV_ERR_BOUNDS in the call's error word, and the kernel goes on, so the context stays usable.
// A stand-in for a memory checker where none can be run. In a normal build sv_ldg is __ldg,
// sv_ld a plain load, sv_st a plain store, and no check exists.
#ifdef SV_DEBUG_BOUNDS
constexpr int kDbgRanges = 32;
struct DbgRanges {
    unsigned long long lo[kDbgRanges], hi[kDbgRanges];  // [lo, hi) byte ranges
    int n;
    unsigned *flags;  // the call's error word pair (bit SV_ERR_BOUNDS goes to flags[1])
};
__device__ DbgRanges g_dbg;

__device__ __noinline__ bool dbg_ok(const void *p, unsigned bytes)
{
    const unsigned long long a = reinterpret_cast<unsigned long long>(p);
    for (int k = 0; k < g_dbg.n; ++k)
        if (a >= g_dbg.lo[k] && a + bytes <= g_dbg.hi[k]) return true;
    if (g_dbg.flags) atomicOr(g_dbg.flags + 1, SV_ERR_BOUNDS);
    return false;
}
#define SV_CHECK(p, bytes) dbg_ok((p), (bytes))
#else
#define SV_CHECK(p, bytes) true
#endif

template <typename T>
__device__ __forceinline__ T sv_ldg(const T *p)
{
    if (!SV_CHECK(p, sizeof(T))) return T{};
    return __ldg(p);
}
template <typename T>
__device__ __forceinline__ T sv_ld(const T *p)
{
    if (!SV_CHECK(p, sizeof(T))) return T{};
    return *p;
}
template <typename T, typename U>
__device__ __forceinline__ void sv_st(T *p, const U &v)
{
    if (SV_CHECK(p, sizeof(T))) *p = v;
}

// ---------------------------------------------------------------------------------------
// element loads
// ---------------------------------------------------------------------------------------
template <typename T> struct Elem;
template <> struct Elem<float> {
    static __device__ __forceinline__ float at(const float *p, size_t k) { return sv_ldg(p + k); }
};
template <> struct Elem<uint16_t> {
    static __device__ __forceinline__ float at(const uint16_t *p, size_t k)
    {
        return __uint_as_float(static_cast<uint32_t>(sv_ldg(p + k)) << 16);
    }
};

// Programmatic dependent launch: a statistics CTA lets the verify grid be scheduled once every
// statistics CTA is running (griddepcontrol.launch_dependents); the verify kernel, after a
// prologue that reads only inputs, waits there until the statistics grid has completed and its
// writes are visible (griddepcontrol.wait; returns at once without such a predecessor).
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint4 ldg_v4(const void *p)
{
    return sv_ldg(reinterpret_cast<const uint4 *>(p));
}

// ---------------------------------------------------------------------------------------
// race keys
// ---------------------------------------------------------------------------------------
// Keys as order-preserving unsigned integers. A candidate is packed as (key, ~v) into 64 bits,
// so that the largest packed value is the largest key with the lowest index among equal keys;
// 0 means no candidate (every finite or infinite key encodes above 0).
__device__ __forceinline__ unsigned key_enc(float f)
{
    const unsigned b = __float_as_uint(f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_dec(unsigned e)
{
    return __uint_as_float((e & 0x80000000u) ? (e & 0x7FFFFFFFu) : ~e);
}
__device__ __forceinline__ unsigned long long pack_key(float key, int v)
{
    return (static_cast<unsigned long long>(key_enc(key)) << 32) |
           static_cast<unsigned>(~static_cast<unsigned>(v));
}
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long p)
{
    const unsigned hi = static_cast<unsigned>(p >> 32);
    const unsigned mh = __reduce_max_sync(0xFFFFFFFFu, hi);
    const unsigned ml = __reduce_max_sync(0xFFFFFFFFu, hi == mh ? static_cast<unsigned>(p) : 0u);
    return (static_cast<unsigned long long>(mh) << 32) | ml;
}

// Upper bound of every key whose weight is at most exp(y) for the y that gave b = exp(y) / E:
// covers a possible few-ulp non-monotonicity of the binary32 exp, with a wide margin (keys are
// >= 0; divisions round monotonically).
__device__ __forceinline__ float key_bound(float b) { return b * 1.00002f; }

__device__ __forceinline__ void emit_row(int i, int jstar, int K, int q0, int token,
                                         const int32_t *__restrict__ draft_ids,
                                         int32_t *__restrict__ sampled, int stride,
                                         int32_t *__restrict__ num_sampled,
                                         int32_t *__restrict__ num_rejected, int tid, int nthreads)
{
    int32_t *out = sampled + static_cast<size_t>(i) * stride;
    for (int s = tid; s < stride; s += nthreads)
        sv_st(out + s, s < jstar ? sv_ld(draft_ids + q0 + s) : (s == jstar ? token : -1));
    if (tid == 0) {
        sv_st(num_sampled + i, jstar + 1);
        sv_st(num_rejected + i, jstar < 0 ? 0 : K - jstar);
    }
}

// ---------------------------------------------------------------------------------------
// requests
// ---------------------------------------------------------------------------------------
// Request of logit row r: the largest i in [0, n) with cu[i] + i <= r (request i owns rows
// cu[i] + i .. cu[i + 1] + i); with draft_rows, of draft row r: the largest i with cu[i] <= r
// (request i owns draft rows cu[i] .. cu[i + 1] - 1). A 32-way search by one full warp; the result
// stays in [0, n) whatever cu holds.
__device__ __forceinline__ int row_request(const int32_t *__restrict__ cu, int n, int r, int lane,
                                           bool draft_rows = false)
{
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) >> 5;
        const int p = lo + lane * step;
        const bool ok = lane == 0 || (p < hi && sv_ldg(cu + p) + (draft_rows ? 0 : p) <= r);
        const unsigned b = __ballot_sync(0xFFFFFFFFu, ok);
        lo += (31 - __clz(b)) * step;
        hi = min(hi, lo + step);
    }
    return lo;
}

// 1 / T of request i, or 1 for a greedy request (flag set, or !(T > 0)).
struct RequestTable {
    const int32_t *cu;
    const float *temperature;
    const uint8_t *is_greedy;
    const int32_t *top_k;  // or nullptr; top_k == 1 keeps only the largest logit: greedy
    int n;
};

// 1 / T of request i, 1 for a greedy request: flag set, T <= 0 ([spec-in-vllm] 7.0.1;
// [mini-sglang] T <= 0) or top_k == 1 ([mini-sglang]: only the largest logit is kept).
__device__ __forceinline__ float request_invT(const RequestTable &rq, int i, bool &greedy)
{
    const float T = sv_ldg(rq.temperature + i);
    greedy = sv_ldg(rq.is_greedy + i) != 0 || !(T > 0.0f) || (rq.top_k && sv_ldg(rq.top_k + i) == 1);
    return greedy ? 1.0f : __frcp_rn(T);
}

// ---------------------------------------------------------------------------------------
// logits processors: the frequency penalty ([MTP-eagle] 其他 / 重复惩罚: logit -= penalty *
// output_bin_counts), applied before the temperature and the softmax ([spec-notes] 8.2)
// ---------------------------------------------------------------------------------------
struct PenTable {
    const float *f;             // [n] frequency penalty, or nullptr (no penalty)
    const int32_t *counts;      // [counts_rows, V] output token counts
    const int32_t *counts_row;  // [n] counts row of each request, or nullptr (row i)
    int counts_rows;
    int nd;                     // draft tokens of the batch (length of draft_ids)
    int kmax;                   // most drafts of one request
    const uint32_t *mask;       // [n][mask_stride] nonzero bits of each request's counts, or nullptr
    int mask_stride;            // words per request: ceil(V / 32) + 1 (a zero word last)
};

// The penalty of one logit row: y_v = fma(-f, c_v, l_v) where f != 0 and c_v != 0, else l_v;
// c_v = the request's count of v plus the drafts before this position equal to v (the target
// conditions on them there).
struct PenRow {
    float f;               // 0: no penalty
    const int32_t *cnt;    // the request's counts row
    const int32_t *prev;   // drafts before this position
    int nprev;
    const uint32_t *mask;  // the counts row's nonzero bits (sv_pen_mask_kernel), or nullptr
};

// Request i, position j (drafts from q0). A counts row outside [0, counts_rows) gives no penalty
// (and is reported by the verify kernel). The statistics and selection kernels run before the
// verify kernel has checked cu_num_draft, so q0 and j come from unchecked device data there:
// a position whose earlier drafts would lie outside draft_ids[0, nd) gets no penalty either
// (such a batch emits nothing, by the verify kernel's check).
__device__ __forceinline__ PenRow pen_row(const PenTable &pt, const int32_t *draft_ids, int i,
                                          int q0, int j, int V)
{
    PenRow r{0.0f, nullptr, nullptr, 0};
    if (!pt.f) return r;
    if (q0 < 0 || q0 > pt.nd || j < 0 || j > pt.kmax || j > pt.nd - q0) return r;
    const int crow = pt.counts_row ? sv_ldg(pt.counts_row + i) : i;
    if (crow < 0 || crow >= pt.counts_rows) return r;
    r.f = sv_ldg(pt.f + i);
    r.cnt = pt.counts + static_cast<size_t>(crow) * V;
    r.prev = draft_ids + q0;
    r.nprev = j;
    r.mask = pt.mask ? pt.mask + static_cast<size_t>(i) * pt.mask_stride : nullptr;
    return r;
}

__device__ __forceinline__ bool pen_counts_row_bad(const PenTable &pt, int i)
{
    if (!pt.f) return false;
    const int crow = pt.counts_row ? sv_ldg(pt.counts_row + i) : i;
    return crow < 0 || crow >= pt.counts_rows;
}

__device__ __forceinline__ float pen_apply(const PenRow &r, float l, int v)
{
    if (r.f == 0.0f) return l;
    int c = sv_ldg(r.cnt + v);
    for (int k = 0; k < r.nprev; ++k) c += sv_ldg(r.prev + k) == v;
    return c == 0 ? l : __fmaf_rn(-r.f, __int2float_rn(c), l);
}

// bf16 upper bound of an fp32 value (rounded toward +inf), for line maxima of penalised rows.
__device__ __forceinline__ uint16_t bf16_round_up(float v)
{
    const uint32_t u = __float_as_uint(v);
    if ((u & 0xFFFFu) == 0u || v != v) return static_cast<uint16_t>(u >> 16);
    return static_cast<uint16_t>((u >> 31) ? (u >> 16) : (u >> 16) + 1u);
}

// ---------------------------------------------------------------------------------------
// 1. row statistics
// ---------------------------------------------------------------------------------------
struct OnlineMax {
    float L = -kInf;   // running max of raw logits
    float s = 0.0f;    // running sum of 2^((l - L) c)
    float Ls = 0.0f;   // the shift: L once L is finite (0 before, so that -inf logits add 2^-inf = 0)
    int best_e = -1;   // element where L was first reached (scalar path), or -1
    int best_p = -1;   // pair where L was first reached (vector path), or -1
};

// Fold one logit at index e (head / tail of a segment; indices increase).
__device__ __forceinline__ void fold1(OnlineMax &st, float l, int e, float c)
{
    if (l > st.L) {
        st.s = st.s == 0.0f ? 0.0f : st.s * sv::ex2_approx((st.L - l) * c);
        st.L = l;
        st.Ls = l;
        st.best_e = e;
        st.best_p = -1;
    }
    // 2^((l - L) c): the difference first, so that a large L c loses nothing to rounding
    st.s += sv::ex2_approx((l - st.Ls) * c);
}

// The statistics kernel streams 64-byte pairs: two 32-byte loads per lane and round, the lanes of
// a warp on consecutive pairs (a 2 KB stretch per warp).
constexpr int kPairBytes = 64;

__device__ __forceinline__ void ldg_pair(const char *p, uint32_t (&w)[16])
{
    if (!SV_CHECK(p, kPairBytes)) {
#pragma unroll
        for (int k = 0; k < 16; ++k) w[k] = 0u;
        return;
    }
    asm("ld.global.nc.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]), "=r"(w[6]),
          "=r"(w[7])
        : "l"(p));
    asm("ld.global.nc.v8.u32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
        : "=r"(w[8]), "=r"(w[9]), "=r"(w[10]), "=r"(w[11]), "=r"(w[12]), "=r"(w[13]), "=r"(w[14]),
          "=r"(w[15])
        : "l"(p + 32));
}

// Element h of a pair (bf16: the low half of word h / 2 first).
template <typename T>
__device__ __forceinline__ float pair_elem(const uint32_t (&w)[16], int h)
{
    if constexpr (sizeof(T) == 2)
        return __uint_as_float((h & 1) ? (w[h >> 1] & 0xFFFF0000u) : (w[h >> 1] << 16));
    else
        return __uint_as_float(w[h]);
}

// Largest element of a pair in a form that combines cheaply (bf16: max.bf16x2 over the words,
// two candidates per word; fp32: a float), and the largest over the lanes that share a
// 64-element line (2 consecutive lanes for bf16, 4 for fp32; every lane must take part).
template <typename T> struct PairMax;
template <> struct PairMax<uint16_t> {
    using P = uint32_t;
    static constexpr int kLanes = 2;
    static __device__ __forceinline__ P max2(P a, P b)
    {
        P d;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    static __device__ __forceinline__ P of(const uint32_t (&w)[16])
    {
        P m[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m[k] = max2(w[2 * k], w[2 * k + 1]);
#pragma unroll
        for (int k = 0; k < 4; ++k) m[k] = max2(m[2 * k], m[2 * k + 1]);
        return max2(max2(m[0], m[1]), max2(m[2], m[3]));
    }
    static __device__ __forceinline__ P none() { return 0xFF80FF80u; }
    static __device__ __forceinline__ float value(P m)
    {
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
    }
    static __device__ __forceinline__ P line(P m)
    {
        return max2(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
    }
    static __device__ __forceinline__ uint16_t store(P m)  // a bf16 value: exact
    {
        return static_cast<uint16_t>(__float_as_uint(value(m)) >> 16);
    }
};
template <> struct PairMax<float> {
    using P = float;
    static constexpr int kLanes = 4;
    static __device__ __forceinline__ P max2(P a, P b) { return fmaxf(a, b); }
    static __device__ __forceinline__ P of(const uint32_t (&w)[16])
    {
        float m[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) m[k] = fmaxf(__uint_as_float(w[2 * k]), __uint_as_float(w[2 * k + 1]));
#pragma unroll
        for (int k = 0; k < 4; ++k) m[k] = fmaxf(m[2 * k], m[2 * k + 1]);
        return fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3]));
    }
    static __device__ __forceinline__ P none() { return -kInf; }
    static __device__ __forceinline__ float value(P m) { return m; }
    static __device__ __forceinline__ P line(P m)
    {
        m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
        return fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
    }
    static __device__ __forceinline__ float store(P m) { return m; }
};

// Two fp32 values in one 64-bit register pair, and the packed fp32x2 operations of sm_100+
// (each lane an ordinary correctly rounded add / multiply).
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}
__device__ __forceinline__ unsigned long long f2_mul(unsigned long long a, unsigned long long b)
{
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Elements 2k and 2k + 1 of a pair as an fp32x2 value.
template <typename T>
__device__ __forceinline__ unsigned long long pair_elems2(const uint32_t (&w)[16], int k)
{
    if constexpr (sizeof(T) == 2)
        return f2_pack(__uint_as_float(w[k] << 16), __uint_as_float(w[k] & 0xFFFF0000u));
    else
        return f2_pack(__uint_as_float(w[2 * k]), __uint_as_float(w[2 * k + 1]));
}

// Fold pair p, whose largest element is mx, without branches: one rescale of the running sum,
// then the sum of 2^((l - L) c), two elements per packed add, multiply and add (the difference
// is taken before the scaling: l c - L c would lose the low bits of a large L c). Only the pair that first
// reached the max is recorded; its lowest index is recovered at the end of the segment.
template <typename T>
__device__ __forceinline__ void fold_pair(OnlineMax &st, const uint32_t (&w)[16], int p, float c,
                                          float mx)
{
    constexpr int kPE = kPairBytes / sizeof(T);
    const bool up = mx > st.L;
    st.s *= sv::ex2_approx(up ? (st.L - mx) * c : 0.0f);  // L = -inf: 2^-inf = 0 (s was 0)
    st.best_p = up ? p : st.best_p;
    st.best_e = up ? -1 : st.best_e;
    st.L = up ? mx : st.L;
    st.Ls = st.L > -kInf ? st.L : 0.0f;
    const unsigned long long c2 = f2_pack(c, c), nL2 = f2_pack(-st.Ls, -st.Ls);
    unsigned long long acc[2] = {0ull, 0ull};  // fp32x2 zeros
#pragma unroll
    for (int k = 0; k < kPE / 2; ++k) {
        float y0, y1;
        f2_unpack(f2_mul(f2_add(pair_elems2<T>(w, k), nL2), c2), y0, y1);
        acc[k & 1] = f2_add(acc[k & 1], f2_pack(sv::ex2_approx(y0), sv::ex2_approx(y1)));
    }
    float a0, a1, b0, b1;
    f2_unpack(acc[0], a0, a1);
    f2_unpack(acc[1], b0, b1);
    st.s += (a0 + b0) + (a1 + b1);
}

// fold_pair over values already processed (the penalty path): the same steps on y[0..n).
template <int n>
__device__ __forceinline__ void fold_vals(OnlineMax &st, const float (&y)[n], int p, float c,
                                          float mx)
{
    const bool up = mx > st.L;
    st.s *= sv::ex2_approx(up ? (st.L - mx) * c : 0.0f);
    st.best_p = up ? p : st.best_p;
    st.best_e = up ? -1 : st.best_e;
    st.L = up ? mx : st.L;
    st.Ls = st.L > -kInf ? st.L : 0.0f;
    const unsigned long long c2 = f2_pack(c, c), nL2 = f2_pack(-st.Ls, -st.Ls);
    unsigned long long acc[2] = {0ull, 0ull};
#pragma unroll
    for (int k = 0; k < n / 2; ++k) {
        float y0, y1;
        f2_unpack(f2_mul(f2_add(f2_pack(y[2 * k], y[2 * k + 1]), nL2), c2), y0, y1);
        acc[k & 1] = f2_add(acc[k & 1], f2_pack(sv::ex2_approx(y0), sv::ex2_approx(y1)));
    }
    float a0, a1, b0, b1;
    f2_unpack(acc[0], a0, a1);
    f2_unpack(acc[1], b0, b1);
    st.s += (a0 + b0) + (a1 + b1);
}

// Division by a launch constant d > 0 without a division instruction: with M = ceil(2^64 / d)
// (0 stands for d = 1), floor(a * M / 2^64) is floor(a / d) or one more for 0 <= a < 2^63, and
// one multiply decides which.
struct Divisor {
    long long d;
    unsigned long long magic;
};
__host__ inline Divisor make_divisor(long long d)
{
    return Divisor{d, d == 1 ? 0ull : ~0ull / static_cast<unsigned long long>(d) + 1ull};
}
__device__ __forceinline__ long long div_floor(long long a, const Divisor &q)
{
    if (q.magic == 0ull) return a;
    long long r = static_cast<long long>(__umul64hi(static_cast<unsigned long long>(a), q.magic));
    if (r * q.d > a) --r;
    return r;
}

// Largest element of a 16-byte vector in a form that combines cheaply (bf16: two halves packed
// in a word, max.bf16x2; fp32: a float), and the largest over the lanes that share a 64-element
// line (8 consecutive lanes for bf16, 16 for fp32, aligned to that in the warp; every lane of the
// warp must take part).
template <typename T> struct VecMax;
template <> struct VecMax<uint16_t> {
    using P = uint32_t;
    static constexpr int kLanes = 8;
    static __device__ __forceinline__ P max2(P a, P b)
    {
        P d;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
        return d;
    }
    static __device__ __forceinline__ P of(const uint4 &w) { return max2(max2(w.x, w.y), max2(w.z, w.w)); }
    static __device__ __forceinline__ P none() { return 0xFF80FF80u; }
    static __device__ __forceinline__ float value(P m)
    {
        return fmaxf(__uint_as_float(m << 16), __uint_as_float(m & 0xFFFF0000u));
    }
    static __device__ __forceinline__ P line(P m)
    {
#pragma unroll
        for (int o = 1; o < kLanes; o <<= 1) m = max2(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        return m;
    }
    static __device__ __forceinline__ uint16_t store(P m)  // a bf16 value: exact
    {
        return static_cast<uint16_t>(__float_as_uint(value(m)) >> 16);
    }
};
template <> struct VecMax<float> {
    using P = float;
    static constexpr int kLanes = 16;
    static __device__ __forceinline__ P max2(P a, P b) { return fmaxf(a, b); }
    static __device__ __forceinline__ P of(const uint4 &w)
    {
        return fmaxf(fmaxf(__uint_as_float(w.x), __uint_as_float(w.y)),
                     fmaxf(__uint_as_float(w.z), __uint_as_float(w.w)));
    }
    static __device__ __forceinline__ P none() { return -kInf; }
    static __device__ __forceinline__ float value(P m) { return m; }
    static __device__ __forceinline__ P line(P m)
    {
#pragma unroll
        for (int o = 1; o < kLanes; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        return m;
    }
    static __device__ __forceinline__ float store(P m) { return m; }
};

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

// Warp reduction of (L, s, idx); the result is valid in every lane.
__device__ __forceinline__ void warp_reduce_stat(float &L, float &s, int &idx, float c)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float L2 = __shfl_xor_sync(0xFFFFFFFFu, L, o);
        const float s2 = __shfl_xor_sync(0xFFFFFFFFu, s, o);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, idx, o);
        combine_stat(L, s, idx, L2, s2, i2, c);
    }
}

// Segment [b, e) of row `row`, by the whole CTA without any barrier: the elements before the
// first 64-element line boundary one by one, then 64-byte pairs, one per lane and round, then the
// last few elements one by one. Every warp looks the row's request up itself (while its first
// round is in flight) and publishes its own partial statistics of the segment, at
// part[(row * maxseg + seg) * kWarps + warp]. With `s_lines`, the largest logit of every line that
// the pairs cover completely is stored at s_lines[line - line_base] in shared memory (line =
// (base_off + flattened element) / 64).
template <typename T>
__device__ __forceinline__ void stats_segment(const T *__restrict__ logits, int V, int row, int b,
                                              int e, int seg, int maxseg, int base_off,
                                              const RequestTable &rq, StatPart *__restrict__ part,
                                              T *__restrict__ s_lines, long long line_base,
                                              bool draft_rows)
{
    const long long rbase = static_cast<long long>(row) * V;
    const T *rp = logits + rbase;
    constexpr int kPE = kPairBytes / sizeof(T);  // elements per pair
    constexpr int kPPL = PairMax<T>::kLanes;     // pairs per line
    const long long pos_b = base_off + rbase + b;  // line coordinate of element b
    const int head = static_cast<int>((kGroup - (pos_b & (kGroup - 1))) & (kGroup - 1));
    const int a0 = min(e, b + head);  // on a line boundary: 64-element aligned in memory
    const int npair = (e - a0) / kPE;
    const int a1 = a0 + npair * kPE;
    const char *pbase = reinterpret_cast<const char *>(rp + a0);
    const int line0 = static_cast<int>(((pos_b + (a0 - b)) >> 6) - line_base);  // pair 0's line
    const int lane = threadIdx.x & 31;

    // the warp's pairs of a round start at ub: every lane runs the same rounds; the pair of the
    // round after next is requested before the current one is folded (three register buffers in
    // rotation: two rounds in flight while one is folded)
    int ub = static_cast<int>(threadIdx.x) & ~31;
    uint32_t w0[16], w1[16], w2[16];
    if (ub + lane < npair) ldg_pair(pbase + static_cast<size_t>(ub + lane) * kPairBytes, w0);
    if (ub + lane + kThreads < npair)
        ldg_pair(pbase + static_cast<size_t>(ub + lane + kThreads) * kPairBytes, w1);
    bool greedy;
    const float c = request_invT(rq, row_request(rq.cu, rq.n, row, lane, draft_rows), greedy) * kLog2e;

    OnlineMax st;
    for (int ee = b + threadIdx.x; ee < a0; ee += kThreads) fold1(st, Elem<T>::at(rp, ee), ee, c);
    auto round = [&](const uint32_t (&cur)[16], uint32_t (&nxt)[16]) {
        const int p = ub + lane;
        const bool valid = p < npair;
        if (p + 2 * kThreads < npair)
            ldg_pair(pbase + static_cast<size_t>(p + 2 * kThreads) * kPairBytes, nxt);
        const typename PairMax<T>::P pm = valid ? PairMax<T>::of(cur) : PairMax<T>::none();
        if (s_lines) {
            const typename PairMax<T>::P lm = PairMax<T>::line(pm);
            if ((lane & (kPPL - 1)) == 0 && p + kPPL - 1 < npair)
                s_lines[line0 + p / kPPL] = PairMax<T>::store(lm);
        }
        if (valid) fold_pair<T>(st, cur, p, c, PairMax<T>::value(pm));
        ub += kThreads;
    };
    while (ub < npair) {
        round(w0, w2);
        if (ub >= npair) break;
        round(w1, w0);
        if (ub >= npair) break;
        round(w2, w1);
    }
    for (int ee = a1 + threadIdx.x; ee < e; ee += kThreads) fold1(st, Elem<T>::at(rp, ee), ee, c);

    // where this thread's max first occurs: an element, or the pair that first reached it
    int idx = st.best_e >= 0 ? argmax_candidate(st.best_e, false) : INT_MAX;
    if (st.best_p >= 0) idx = argmax_candidate(a0 + st.best_p * kPE, true);
    float L = st.L, s = st.s;
    warp_reduce_stat(L, s, idx, c);
    if (lane == 0)
        sv_st(part + (static_cast<size_t>(row) * maxseg + seg) * kWarps + (threadIdx.x >> 5), StatPart{L, s, idx, 0});
}

// stats_segment for the rows of a batch with a frequency penalty, over the processed values y
// (see pen_apply): the plain path's pair stream, each pair requested with the two words of the
// row's counts mask (sv_pen_mask_kernel) that hold its tokens' bits. A pair's counted tokens
// (count bits, and earlier drafts) are set to -inf in its buffer and the pair is folded as raw
// logits, which its other tokens' values are; the counted ones, few since counts are sparse,
// then take their counts and drafts one by one (y = l - f n, as pen_apply). A maximum of a pair
// with counted tokens is recorded by its exact index (a reader can only resolve a pair of raw
// values). A row without a penalty (or a draft row) has no mask and no drafts: every pair folds
// as raw logits. Line maxima are those of y rounded up to the logits' type: upper bounds.
template <typename T>
__device__ __forceinline__ void stats_segment_mask(const T *__restrict__ logits, int V, int row, int b,
                                                   int e, int seg, int maxseg, int base_off,
                                                   const RequestTable &rq, const PenTable &pt,
                                                   const int32_t *__restrict__ draft_ids,
                                                   bool draft_rows, StatPart *__restrict__ part,
                                                   T *__restrict__ s_lines, long long line_base)
{
    const long long rbase = static_cast<long long>(row) * V;
    const T *rp = logits + rbase;
    constexpr int kPE = kPairBytes / sizeof(T);  // elements per pair
    constexpr int kPPL = PairMax<T>::kLanes;     // pairs per line
    const long long pos_b = base_off + rbase + b;
    const int head = static_cast<int>((kGroup - (pos_b & (kGroup - 1))) & (kGroup - 1));
    const int a0 = min(e, b + head);
    const int npair = (e - a0) / kPE;
    const int a1 = a0 + npair * kPE;
    const char *pbase = reinterpret_cast<const char *>(rp + a0);
    const int line0 = static_cast<int>(((pos_b + (a0 - b)) >> 6) - line_base);
    const int lane = threadIdx.x & 31;
    int ub = static_cast<int>(threadIdx.x) & ~31;
    uint32_t w0[16], w1[16], w2[16];
    if (ub + lane < npair) ldg_pair(pbase + static_cast<size_t>(ub + lane) * kPairBytes, w0);
    if (ub + lane + kThreads < npair)
        ldg_pair(pbase + static_cast<size_t>(ub + lane + kThreads) * kPairBytes, w1);
    // the row's request and penalty, while the first rounds are in flight
    const int i = row_request(rq.cu, rq.n, row, lane, draft_rows);
    PenRow pr{0.0f, nullptr, nullptr, 0, nullptr};
    if (!draft_rows) {
        const int q0 = sv_ldg(rq.cu + i);
        pr = pen_row(pt, draft_ids, i, q0, row - q0 - i, V);
        if (pr.f == 0.0f) pr = PenRow{0.0f, nullptr, nullptr, 0, nullptr};
    }
    bool greedy;
    const float c = request_invT(rq, i, greedy) * kLog2e;
    const int np = pr.nprev;
    const int pv = lane < np ? sv_ldg(pr.prev + lane) : -1;  // earlier drafts: lane k the k-th

    // the mask words of pair p's tokens [t, t + kPE): word t / 32 and the next (at most the zero
    // word after the row's last, since t + kPE <= V)
    auto load_mask = [&](int p, uint2 &m) {
        if (!pr.mask) return;
        const int t = a0 + p * kPE;
        m.x = sv_ldg(pr.mask + (t >> 5));
        m.y = sv_ldg(pr.mask + (t >> 5) + 1);
    };
    auto load = [&](int p, uint32_t (&w)[16], uint2 &m) {
        ldg_pair(pbase + static_cast<size_t>(p) * kPairBytes, w);
        load_mask(p, m);
    };
    auto drafts_at = [&](int v) {  // how many earlier drafts are token v
        int n = 0;
        for (int k = 0; k < np; ++k) n += sv_ldg(pr.prev + k) == v;
        return n;
    };
    uint2 m0 = make_uint2(0u, 0u), m1 = m0, m2 = m0;
    if (ub + lane < npair) load_mask(ub + lane, m0);
    if (ub + lane + kThreads < npair) load_mask(ub + lane + kThreads, m1);

    OnlineMax st;
    for (int ee = b + threadIdx.x; ee < a0; ee += kThreads)
        fold1(st, pen_apply(pr, Elem<T>::at(rp, ee), ee), ee, c);
    // round: fold pair p of `cur` (modified in place: the buffer is reloaded only in the next
    // round) and request the pair two rounds ahead into `nxt`
    auto round = [&](uint32_t (&cur)[16], const uint2 &mc, uint32_t (&nxt)[16], uint2 &mn) {
        const int p = ub + lane;
        const bool valid = p < npair;
        if (p + 2 * kThreads < npair) load(p + 2 * kThreads, nxt, mn);
        const int t = a0 + p * kPE;
        const int wlo = a0 + ub * kPE;  // the warp's tokens this round: [wlo, wlo + 32 kPE)
        const bool scan = np > 32 || __ballot_sync(0xFFFFFFFFu, static_cast<unsigned>(pv - wlo) <
                                                                    static_cast<unsigned>(32 * kPE)) != 0u;
        // the pair's counted tokens (count bits, and earlier drafts in scan rounds)
        const int sh = t & 31;
        uint32_t bits = mc.x >> sh;
        if (sh) bits |= mc.y << (32 - sh);
        if constexpr (kPE < 32) bits &= (1u << kPE) - 1u;
        uint32_t xb = valid ? bits : 0u;
        if (scan && valid)
            for (int k = 0; k < np; ++k) {
                const unsigned d = static_cast<unsigned>(sv_ldg(pr.prev + k) - t);
                if (d < static_cast<unsigned>(kPE)) xb |= 1u << d;
            }
        // the others fold as raw logits: the counted ones are set to -inf in the buffer first
        if (xb) {
#pragma unroll
            for (int jw = 0; jw < 16; ++jw) {
                if constexpr (sizeof(T) == 2) {
                    const uint32_t b2 = (xb >> (2 * jw)) & 3u;
                    const uint32_t m = ((b2 & 1u) ? 0x0000FFFFu : 0u) | ((b2 & 2u) ? 0xFFFF0000u : 0u);
                    cur[jw] = (cur[jw] & ~m) | (0xFF80FF80u & m);
                } else {
                    if ((xb >> jw) & 1u) cur[jw] = 0xFF800000u;
                }
            }
        }
        const typename PairMax<T>::P pm = valid ? PairMax<T>::of(cur) : PairMax<T>::none();
        float lmv = PairMax<T>::value(pm);  // the pair's largest processed value
        if (valid) {
            const float L0 = st.L;
            fold_pair<T>(st, cur, p, c, lmv);
            if (xb && st.L != L0) {  // a new maximum among raw values next to counted ones:
                int hh = kPE - 1;     // a reader could not tell them apart, so the exact index
#pragma unroll
                for (int h = kPE - 1; h >= 0; --h)
                    if (pair_elem<T>(cur, h) == st.L) hh = h;
                st.best_e = t + hh;
                st.best_p = -1;
            }
        }
        // the counted tokens one by one (a tie with a maximum inside this pair keeps the lower
        // index; an earlier pair's maximum has a lower index than any of them)
        while (xb) {
            const int k = __ffs(xb) - 1;
            xb &= xb - 1u;
            const int v = t + k;
            const float l = Elem<T>::at(rp, v);
            int n = (bits >> k) & 1u ? sv_ldg(pr.cnt + v) : 0;
            if (scan) n += drafts_at(v);
            const float y = n == 0 ? l : __fmaf_rn(-pr.f, __int2float_rn(n), l);
            if (y > st.L) {
                st.s = st.s == 0.0f ? 0.0f : st.s * sv::ex2_approx((st.L - y) * c);
                st.L = y;
                st.Ls = y;
                st.best_e = v;
                st.best_p = -1;
            } else if (y == st.L && st.best_e >= t && v < st.best_e) {
                st.best_e = v;
            }
            st.s += sv::ex2_approx((y - st.Ls) * c);
            lmv = fmaxf(lmv, y);
        }
        if (s_lines) {
            float lm = lmv;
#pragma unroll
            for (int o = 1; o < kPPL; o <<= 1) lm = fmaxf(lm, __shfl_xor_sync(0xFFFFFFFFu, lm, o));
            if ((lane & (kPPL - 1)) == 0 && p + kPPL - 1 < npair) {
                if constexpr (sizeof(T) == 2) s_lines[line0 + p / kPPL] = bf16_round_up(lm);
                else s_lines[line0 + p / kPPL] = lm;
            }
        }
        ub += kThreads;
    };
    while (ub < npair) {
        round(w0, m0, w2, m2);
        if (ub >= npair) break;
        round(w1, m1, w0, m0);
        if (ub >= npair) break;
        round(w2, m2, w1, m1);
    }
    for (int ee = a1 + threadIdx.x; ee < e; ee += kThreads)
        fold1(st, pen_apply(pr, Elem<T>::at(rp, ee), ee), ee, c);

    int idx = st.best_e >= 0 ? argmax_candidate(st.best_e, false) : INT_MAX;
    if (st.best_p >= 0) idx = argmax_candidate(a0 + st.best_p * kPE, true);
    float L = st.L, s = st.s;
    warp_reduce_stat(L, s, idx, c);
    if (lane == 0)
        sv_st(part + (static_cast<size_t>(row) * maxseg + seg) * kWarps + (threadIdx.x >> 5), StatPart{L, s, idx, 0});
}

// One [rows x V] array the statistics kernel streams: the target logits, or the draft logits of
// the draft-logits mode (rows = draft tokens, each belonging to the request that drafted it).
template <typename T>
struct StatsArray {
    const T *logits;
    long long total;     // rows * V
    Divisor chunk, dv;   // elements per CTA; V
    int base_off;        // (address mod 64 elements) / element size
    int grid;            // CTAs of this array
    int draft_rows;      // row r is draft row r (request: largest i with cu[i] <= r)
    StatPart *part;      // [rows x maxseg x kWarps] partials
    T *lines;            // line maxima (target logits only), or nullptr
};

// Row statistics over a flattened [rows x V] array, split evenly: CTA k of an array streams
// elements [k * chunk - base_off, (k + 1) * chunk - base_off) (chunk a multiple of 512, so that
// CTAs meet on line boundaries and own whole 16-byte spans of the line array), which covers one
// or more row segments, and writes one partial per warp and segment. With `lines`, the CTA
// gathers its line maxima in shared memory (chunk / 64 of them) and writes them out at the end in
// one coalesced sweep, lines [k * chunk / 64, (k + 1) * chunk / 64); entries of lines that a row
// covers only in part are left undefined (the verify kernel reads those lines from the logits).
// The first A.grid CTAs take the target logits, the rest the draft logits (if any). Nothing waits
// on another CTA.
// kPen: the batch has a frequency penalty; every row takes stats_segment_mask (one segment
// function per instantiation: the two together need more than a CTA's registers).
template <typename T, bool kPen>
__global__ void __launch_bounds__(kThreads, kPen ? 2 : 3)
sv_stats_kernel(int V, int maxseg, StatsArray<T> A, StatsArray<T> D, RequestTable rq,
                PenTable pt, const int32_t *__restrict__ draft_ids)
{
    extern __shared__ __align__(16) unsigned char s_raw[];
    pdl_launch_dependents();
    const bool second = static_cast<int>(blockIdx.x) >= A.grid;
    const StatsArray<T> X = second ? D : A;
    const int cta = second ? static_cast<int>(blockIdx.x) - A.grid : static_cast<int>(blockIdx.x);
    const long long start = max(0LL, static_cast<long long>(cta) * X.chunk.d - X.base_off);
    const long long stop = min(X.total, static_cast<long long>(cta + 1) * X.chunk.d - X.base_off);
    if (start >= stop) return;
    T *s_lines = X.lines ? reinterpret_cast<T *>(s_raw) : nullptr;
    const long long line_base = static_cast<long long>(cta) * (X.chunk.d >> 6);
    const int r_first = static_cast<int>(div_floor(start, X.dv));
    const int r_last = static_cast<int>(div_floor(stop - 1, X.dv));
    for (int row = r_first; row <= r_last; ++row) {
        const long long rbase = static_cast<long long>(row) * V;
        const int b = static_cast<int>(max(start, rbase) - rbase);
        const int e = static_cast<int>(min(stop, rbase + V) - rbase);
        const int fk = static_cast<int>(div_floor(X.base_off + rbase, X.chunk));
        if constexpr (kPen)
            stats_segment_mask<T>(X.logits, V, row, b, e, cta - fk, maxseg, X.base_off, rq, pt,
                                  draft_ids, X.draft_rows != 0, X.part, s_lines, line_base);
        else
            stats_segment<T>(X.logits, V, row, b, e, cta - fk, maxseg, X.base_off, rq, X.part,
                             s_lines, line_base, X.draft_rows != 0);
    }
    if (X.lines) {
        __syncthreads();
        const long long lines_end = (X.base_off + X.total + kGroup - 1) >> 6;
        const int nl = static_cast<int>(min(X.chunk.d >> 6, lines_end - line_base));
        const int nv = nl * static_cast<int>(sizeof(T)) / 16;  // whole 16-byte vectors
        uint4 *dst = reinterpret_cast<uint4 *>(X.lines + line_base);
        const uint4 *src = reinterpret_cast<const uint4 *>(s_raw);
        for (int k = threadIdx.x; k < nv; k += kThreads) sv_st(dst + k, src[k]);
        for (int k = nv * 16 / static_cast<int>(sizeof(T)) + threadIdx.x; k < nl; k += kThreads)
            sv_st(X.lines + line_base + k, s_lines[k]);
    }
}

// The nonzero pattern of every penalised request's counts row: bit v % 32 of word v / 32 of
// mask[i * stride ..] is set when the count of token v is not 0, and the word after the last is
// 0, so that a pair's two words can be read anywhere in the row. Requests without a penalty, or
// whose counts row is outside the array, are skipped (pen_row gives them no penalty, so nothing
// reads their bits). Each warp writes 32 words: word after word, a coalesced load of its 32
// counts and a ballot. Grid: blocks_per_req CTAs per request, kWarps * 32 words each.
__global__ void __launch_bounds__(kThreads)
sv_pen_mask_kernel(PenTable pt, int n, int V, int blocks_per_req, uint32_t *__restrict__ mask)
{
    const int i = static_cast<int>(blockIdx.x) / blocks_per_req;
    if (i >= n) return;
    const int W = pt.mask_stride - 1;  // words of a row before the zero word
    const int wb = (static_cast<int>(blockIdx.x) % blocks_per_req) * (kWarps * 32) +
                   static_cast<int>(threadIdx.x >> 5) * 32;
    if (wb > W) return;  // whole warps
    const float f = sv_ldg(pt.f + i);
    const int crow = pt.counts_row ? sv_ldg(pt.counts_row + i) : i;
    if (f == 0.0f || crow < 0 || crow >= pt.counts_rows) return;
    const int32_t *cnt = pt.counts + static_cast<size_t>(crow) * V;
    const int lane = threadIdx.x & 31;
    uint32_t mine = 0u;  // lane k: word wb + k
#pragma unroll 8
    for (int k = 0; k < 32; ++k) {
        const int v = (wb + k) * 32 + lane;
        const bool nz = v < V && sv_ldg(cnt + v) != 0;
        const uint32_t bw = __ballot_sync(0xFFFFFFFFu, nz);
        if (lane == k) mine = bw;
    }
    if (wb + lane <= W) sv_st(mask + static_cast<size_t>(i) * pt.mask_stride + wb + lane, mine);
}

// ---------------------------------------------------------------------------------------
// 2. verify: acceptance, first rejection, race search, emit
// ---------------------------------------------------------------------------------------
struct VerifyParams {
    RequestTable rq;
    const int32_t *draft_ids;
    const float *q;
    const void *dl;          // draft logits (logits' type), or nullptr
    const StatPart *dpart;   // partials of the draft rows (draft-logits mode)
    Divisor dchunk;          // statistics chunk of the draft logits
    int dbase_off;           // their (address mod 64 elements) / element size
    const StatPart *part;
    uint64_t seed;
    uint32_t req_base;
    int nd, kmax, V, maxseg, base_off;
    Divisor chunk;
    int32_t *sampled, *num_sampled, *num_rejected;
    float *opt_max, *opt_sum;
    int32_t *opt_amax;
    unsigned *flags;
    const uint8_t *partial;      // [n] requests in a chunked prefill, or nullptr
    PenTable pen;                // frequency penalty (pen.f == nullptr: none)
    const float *top_p;          // [n] or nullptr (top_k is in rq)
    const float *sel_tau;        // [rows] thresholds of constrained rows (nullptr: none)
    const float *sel_S;          // [rows] their kept mass
    int nsyn;                    // synthetic acceptance: rates of positions < nsyn (0 = off)
    int f64;                     // race clocks and keys in binary64 (the fp64 Gumbel option)
    float syn[SV_MAX_SYNTHETIC]; // unconditional rate a_j of position j
};

// Synthetic acceptance of draft j ([spec-in-vllm] 7.2 / 7.4): accepted iff the id is valid and
// the conditional rate a_j / a_{j-1} (a_{-1} = 1, 0 once a rate is 0) is >= the position's
// uniform. One thread.
__device__ __forceinline__ bool accept_synthetic(const VerifyParams &P, int j, int qrow,
                                                 uint32_t ireq)
{
    const int d = sv_ldg(P.draft_ids + qrow);
    if (d < 0 || d >= P.V) return false;
    const float a = j < P.nsyn ? P.syn[j] : 0.0f;
    float c = a;
    if (j > 0) {
        const float prev = j - 1 < P.nsyn ? P.syn[j - 1] : 0.0f;
        c = prev > 0.0f ? __fdiv_rn(a, prev) : 0.0f;
    }
    const sv::Philox4 r = sv::philox4x32_10(0u, static_cast<uint32_t>(j), ireq, sv::kTagAccept,
                                            static_cast<uint32_t>(P.seed),
                                            static_cast<uint32_t>(P.seed >> 32));
    return c >= sv::uniform_from_word(r.x);
}

// Acceptance test of draft j ([spec-notes] answer code: draft_prob > 0 and
// target_prob / draft_prob >= uniform; greedy: d == argmax, [spec-notes] 8.3). One thread.
// The inputs of an acceptance test read ahead (before the statistics are complete): the draft
// token, its target logit and its q entry (or draft logit). have == false: read them here.
struct AcceptInputs {
    bool have;
    int d;
    float l, qv;
};

template <typename T>
__device__ __forceinline__ AcceptInputs accept_inputs(const T *rp, int V, int qrow,
                                                      const int32_t *__restrict__ draft_ids,
                                                      const float *__restrict__ q,
                                                      const T *__restrict__ dl)
{
    AcceptInputs a{true, sv_ldg(draft_ids + qrow), 0.0f, 1.0f};
    if (a.d >= 0 && a.d < V) {
        a.l = Elem<T>::at(rp, a.d);
        if (q) a.qv = sv_ldg(q + static_cast<size_t>(qrow) * V + a.d);
        else if (dl) a.qv = Elem<T>::at(dl + static_cast<size_t>(qrow) * V, a.d);
    }
    return a;
}

template <typename T>
__device__ __forceinline__ bool accept_draft(const T *rp, int V, bool greedy, int j, int qrow,
                                             const PenRow &pr, float invT, float m, float S,
                                             float tau, int amax,
                                             const int32_t *__restrict__ draft_ids,
                                             const float *__restrict__ q, const T *__restrict__ dl,
                                             float md, float Sd, uint64_t seed, uint32_t ireq,
                                             AcceptInputs in)
{
    if (!in.have) in = accept_inputs<T>(rp, V, qrow, draft_ids, q, dl);
    const int d = in.d;
    if (greedy) return d == amax;
    if (d < 0 || d >= V) return false;
    const float x_d = __fmul_rn(pen_apply(pr, in.l, d), invT);
    // p' of the constrained target: 0 outside the kept set, S the kept mass
    const float t_d = x_d >= tau ? sv::exp_f32(__fsub_rn(x_d, m)) : 0.0f;
    const float p_d = __fdiv_rn(t_d, S);
    float q_d = 1.0f;
    if (q) {
        q_d = in.qv;
    } else if (dl) {  // q = softmax(draft logits / T), the target's steps on the draft row
        const float xd = __fmul_rn(in.qv, invT);
        q_d = __fdiv_rn(sv::exp_f32(__fsub_rn(xd, md)), Sd);
    }
    const sv::Philox4 r = sv::philox4x32_10(0u, static_cast<uint32_t>(j), ireq, sv::kTagAccept,
                                            static_cast<uint32_t>(seed),
                                            static_cast<uint32_t>(seed >> 32));
    const float u = sv::uniform_from_word(r.x);
    return (q_d > 0.0f) && (__fdiv_rn(p_d, q_d) >= u);
}

// Where a row's elements fall on the 64-element lines of the flattened logits. Flattened
// element e sits on line (base_off + e) / 64, base_off = (address of the array mod 64 elements)
// / element size: a line is 64 elements starting on a 64-element boundary of memory.
struct RowLines {
    long long P0;  // base_off + first flattened element of the row
    long long L0;  // line of the row's first element
    int nl;        // lines the row touches
    int kf, kl;    // first and last line (relative to L0) that lies entirely inside the row
    // line (relative to L0) that holds token v
    __device__ __forceinline__ int of(int v) const { return static_cast<int>(((P0 + v) >> 6) - L0); }
};

__device__ __forceinline__ RowLines row_lines(long long row, int V, int base_off)
{
    RowLines rl;
    rl.P0 = base_off + row * V;
    rl.L0 = rl.P0 >> 6;
    rl.nl = static_cast<int>(((rl.P0 + V - 1) >> 6) - rl.L0) + 1;
    rl.kf = (rl.P0 & (kGroup - 1)) ? 1 : 0;
    rl.kl = ((rl.P0 + V) & (kGroup - 1)) ? rl.nl - 2 : rl.nl - 1;
    return rl;
}

// lm[k] = largest raw logit of the row on line L0 + k (the row's own elements only). The lines
// inside the row come from `lines` (written by the statistics kernel) or, without it, from
// coalesced 16-byte loads of the row; a partial first / last line is read by warp 0 / 1. The
// loads without `lines` take the raw logits, which bound a penalised row only for penalties of
// one sign: launch_all therefore refuses a penalty without a line buffer (the static-scratch
// entry point, the one caller without it, takes no penalty).
template <typename T, bool kPen>
__device__ void row_line_max(const T *__restrict__ rp, int V, const RowLines &rl,
                             const T *__restrict__ lines, float *__restrict__ lm,
                             const PenRow &pr)
{
    constexpr int kVPL = VecMax<T>::kLanes;  // vectors per line
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lines) {
        for (int k = rl.kf + static_cast<int>(threadIdx.x); k <= rl.kl; k += kThreads)
            lm[k] = Elem<T>::at(lines, static_cast<size_t>(rl.L0 + k));
    } else {
        const int nvec = max(0, rl.kl - rl.kf + 1) * kVPL;
        // line L0 + kf starts at token (L0 + kf) * 64 - P0 of the row, on a 16-byte boundary
        const char *lbase = reinterpret_cast<const char *>(rp + ((rl.L0 + rl.kf) * kGroup - rl.P0));
        for (int base = 0; base < nvec; base += 4 * kThreads) {
            uint4 w[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int u = base + static_cast<int>(threadIdx.x) + k * kThreads;
                w[k] = u < nvec ? ldg_v4(lbase + static_cast<size_t>(u) * 16) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float mx = VecMax<T>::value(VecMax<T>::line(VecMax<T>::of(w[k])));
                const int u = base + static_cast<int>(threadIdx.x) + k * kThreads;
                if ((lane & (kVPL - 1)) == 0 && u < nvec) lm[rl.kf + u / kVPL] = mx;
            }
        }
    }
    // partial lines: the first (if the row does not start a line) and the last (if the row does
    // not end one and it is another line)
    int k = -1;
    if (warp == 0 && rl.kf == 1) k = 0;
    if (warp == 1 && rl.kl == rl.nl - 2 && (rl.nl > 1 || rl.kf == 0)) k = rl.nl - 1;
    if (k >= 0) {
        const long long p = (rl.L0 + k) * kGroup;  // first line coordinate of the line
        float mx = -kInf;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const long long v = p + h * 32 + lane - rl.P0;  // token of the row
            if (v >= 0 && v < V) {
                const float l = Elem<T>::at(rp, static_cast<size_t>(v));
                mx = fmaxf(mx, kPen ? pen_apply(pr, l, static_cast<int>(v)) : l);
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        if (lane == 0) lm[k] = mx;
    }
}

// The raced row as the search sees it.
template <typename T>
struct RaceRow {
    const T *rp;        // logits row
    const float *qrow;  // draft distribution row (residual race) or nullptr
    const T *dlrow;     // draft logits row (residual race in draft-logits mode) or nullptr
    PenRow pr;          // the row's frequency penalty
    float tau;          // kept tokens: x >= tau (sampling constraints; -inf: all)
    float md, Sd;       // its max and sum of exponentials
    int V, G;           // vocabulary, groups
    int excl;           // token left out (rejected draft without q), or -1
    float m, S, invT;
    uint32_t j, ireq, k0, k1;  // Philox counter words 1, 2 and key
    uint32_t g0;               // group of the row's token 0 (a vocabulary shard's first group)
    bool f64;                  // race clocks and keys in binary64 (the fp64 Gumbel option)
};

// Shared memory of the search (one CTA). Each warp keeps a queue of candidate tokens (at most
// 32 + 64: it is emptied once it holds 32, and a group adds at most 64).
constexpr int kQueue = 96;
constexpr int kBins = 32;  // candidate bins of the best-first order

struct SearchSmem {
    unsigned long long *buf;  // [sp] candidate entries (key bound, group); shares space with lm
    unsigned long long *tmp;  // [sp] the entries in bin order
    int *bin_n;               // [kBins + 1] entries per bin, then bin starts
    unsigned *bin_max;        // [kBins] largest key bound (encoded) of each bin
    unsigned *top;            // largest group bound (encoded)
    float *lm;                // [G + 2] line maxima of the row, until the bounds are taken
    float *pb;                // [G] upper bound of the group's keys (NaN once evaluated)
    uint32_t *ew;             // [G] word 0 of the group's head call (gives E_g)
    uint8_t *ag;              // [G] slot that holds the group's smallest clock
    unsigned long long *best; // best candidate so far, packed (key, ~v); 0 = none. With binary64
                              // keys: (key rounded down to binary32, ~v), a lower bound that only
                              // prunes; the exact best is kept per warp in wbk / wbv
    unsigned long long *wbk;  // [kWarps] binary64 races: each warp's best key (bits + 1; 0 = none)
    int *wbv;                 // [kWarps] and its token
    int *cnt;
    uint32_t *qgs;            // [kWarps][kQueue] candidate tokens of each warp: group << 6 | slot
    float *ql, *qq;           // [kWarps][kQueue] their raw logits and q entries
};

// Dynamic shared memory layout of a verify CTA (bytes): the candidate buffer (a power of two
// >= G entries of 8 bytes, also holding the G + 2 line maxima), the binned copy of it, m / S /
// argmax of the request's rows and m / S of its draft rows (kmax + 1 each), pb, ew, ag.
struct VerifyLayout {
    size_t tmp, rows, pb, ew, ag, total;
};
__host__ __device__ inline int search_capacity(int G)
{
    int sp = 1;
    while (sp < G) sp <<= 1;
    return sp;
}
__host__ __device__ inline VerifyLayout verify_layout(int V, int kmax)
{
    const size_t G = static_cast<size_t>((V + kGroup - 1) / kGroup);
    const size_t sp = static_cast<size_t>(search_capacity(static_cast<int>(G)));
    VerifyLayout l;
    const size_t buf = 8 * sp > 4 * (G + 2) ? 8 * sp : 4 * (G + 2);
    l.tmp = (buf + 15) / 16 * 16;
    l.rows = l.tmp + 8 * sp;
    l.pb = l.rows + 24 * (static_cast<size_t>(kmax) + 1);  // m, S, argmax, m_d, S_d, tau
    l.ew = l.pb + 4 * G;
    l.ag = l.ew + 4 * G;
    l.total = l.ag + G;
    return l;
}

// Group g's smallest clock, E_g = -log(W) / 64, from word 0 of its head call (exact scaling).
__device__ __forceinline__ float group_emin_word(uint32_t w_head)
{
    return __fmul_rn(-sv::log_f32(sv::uniform_from_word(w_head)), 0x1p-6f);
}

// The group's head uniform W as a binary32 value that is never below it: exact for the binary32
// clocks; for the binary64 ones (52 bits from words 0 and 1) an upper bound from word 0 alone,
// (word 0 + 1) / 2^32 rounded up, which makes -log W and the bounds below only smaller / larger.
__device__ __forceinline__ float head_uniform_ub(uint32_t w0, bool f64)
{
    return f64 ? __fmul_rn(__ull2float_ru(static_cast<unsigned long long>(w0) + 1ull), 0x1p-32f)
               : sv::uniform_from_word(w0);
}

// An upper bound of every key exp(y') / E' with y' <= y and E' >= E_g (W >= the group's head
// uniform, head_uniform_ub), from the hardware approximations: lg2.approx errs by less than 2^-22 absolute and
// ex2.approx by a few 2^-23 relative on these ranges, and the fp32 product y log2(e) by
// |y| 2^-23; the margins below (2^-20 absolute on -log2 W, 2^-12 relative twice) cover all of
// that many times over. Only the evaluation of a group uses its exact E_g. +inf when -log W is
// too small to bound from below (W within about 10^-6 of 1), and for a NaN y.
__device__ __forceinline__ float group_bound(float y, float W)
{
    float l2;
    asm("lg2.approx.f32 %0, %1;" : "=f"(l2) : "f"(W));
    const float nl = (-l2 - 0x1p-20f) * 0x1.62e2p-1f;  // <= -ln W (ln 2 rounded down)
    const float tub = sv::ex2_approx(y * kLog2e) * (1.0f + 0x1p-12f);
    const float b = __fdividef(tub, nl * 0x1p-6f) * (1.0f + 0x1p-12f);
    return (nl > 0.0f && b == b) ? b : kInf;
}

// pb[g] = an upper bound of every key in group g (from x_max = fl(line max * invT) and the
// group's head call), ew[g] / ag[g] = the head's word 0 and slot (binary64 clocks: word 2 gives
// the slot). Returns the thread's best (pb, g) packed, 0 if it has no group.
template <typename T>
__device__ unsigned long long group_bounds(const RaceRow<T> &r, const RowLines &rl,
                                           const SearchSmem &sm)
{
    constexpr int kStep = 4;  // independent groups per thread and step (Philox chains overlap)
    unsigned long long best = 0;
    for (int g0 = threadIdx.x; g0 < r.G; g0 += kStep * kThreads) {
        float lmax[kStep];
        sv::Philox4 h[kStep];
#pragma unroll
        for (int k = 0; k < kStep; ++k) {
            const int g = min(g0 + k * kThreads, r.G - 1);
            const int v0 = g * kGroup, v1 = min(v0 + kGroup, r.V) - 1;
            lmax[k] = fmaxf(sm.lm[rl.of(v0)], sm.lm[rl.of(v1)]);
            h[k] = sv::philox4x32_10(static_cast<uint32_t>(g) + r.g0, r.j, r.ireq,
                                     r.f64 ? sv::kClockHead64 : sv::kClockHead, r.k0, r.k1);
        }
#pragma unroll
        for (int k = 0; k < kStep; ++k) {
            const int g = g0 + k * kThreads;
            if (g < r.G) {
                // a group whose largest x is below the kept set's threshold holds no candidate
                // (x_v = fl(l_v / T) <= fl(lmax / T)): bound 0 (NaN groups stay in the race)
                const float xg = __fmul_rn(lmax[k], r.invT);
                const float b = !(xg < r.tau)
                                    ? group_bound(__fsub_rn(xg, r.m), head_uniform_ub(h[k].x, r.f64))
                                    : 0.0f;
                sm.pb[g] = b;
                sm.ew[g] = h[k].x;
                sm.ag[g] = static_cast<uint8_t>((r.f64 ? h[k].z : h[k].y) & 63u);
                best = max(best, pack_key(b, g));
            }
        }
    }
    return best;
}

__device__ __forceinline__ unsigned long long ld_best(const unsigned long long *s_best)
{
    // one 64-bit shared load, broadcast from lane 0 so that the warp takes one decision
    const unsigned long long v = *reinterpret_cast<const volatile unsigned long long *>(s_best);
    return __shfl_sync(0xFFFFFFFFu, v, 0);
}

// An upper bound of 1 / E_g from W >= the group's head uniform (E_g = -log(W) / 64): hardware
// lg2 and rcp with the margins of group_bound; +inf when -log W is too small to bound from below.
__device__ __forceinline__ float inv_emin_bound(float W)
{
    float l2;
    asm("lg2.approx.f32 %0, %1;" : "=f"(l2) : "f"(W));
    const float nl = (-l2 - 0x1p-20f) * 0x1.62e2p-1f;  // <= -ln W
    return nl > 0.0f ? __frcp_rz(nl * 0x1p-6f) * (1.0f + 0x1p-12f) : kInf;
}

// The binary64 key w / E_v of slot `slot` of group gg (a = the slot of the group's smallest
// clock), with the binary64 clocks of sv_device.cuh.
__device__ __forceinline__ double key_f64(float w, uint32_t gg, int slot, int a, uint32_t j,
                                          uint32_t ireq, uint32_t k0, uint32_t k1)
{
    const sv::Philox4 hd = sv::philox4x32_10(gg, j, ireq, sv::kClockHead64, k0, k1);
    const double E = __dmul_rn(-sv::log_f64(sv::uniform64_from_words(hd.x, hd.y)), 0x1p-6);
    double Ev = E;
    if (slot != a) {
        const sv::Philox4 sl = sv::philox4x32_10(
            gg, j, ireq, sv::kClockHead64 + 1u + static_cast<uint32_t>(slot >> 1), k0, k1);
        const double U = (slot & 1) ? sv::uniform64_from_words(sl.z, sl.w)
                                    : sv::uniform64_from_words(sl.x, sl.y);
        Ev = __dadd_rn(E, -sv::log_f64(U));
    }
    return __ddiv_rn(static_cast<double>(w), Ev);  // >= 0 and finite: E_v >= E_g >= 2^-59
}

// Empty the warp's candidate queue (n entries): one token per lane, its exact weight, its race
// clock and its key, merged into *sm.best. Entry: group g, slot s, raw logit, q entry.
// Slot s = v & 63 of group g: its clock is E_g for the head's slot a, else fl(E_g + (-log U_s)),
// U_s from word s & 3 of slot call s / 4 (tag kClockHead + 1 + s / 4). With binary64 clocks
// (r.f64) the same in double: E_g from the head's words 0 and 1, U_s from words (0, 1) or (2, 3)
// of slot call s / 2 (tag kClockHead64 + 1 + s / 2), the key the binary64 quotient; *sm.best then
// receives the key rounded down (a lower bound, for pruning) and the warp's exact best goes to
// wbk / wbv.
// One queue entry's exact weight (t, or the residual rr; NaN-free, may be <= 0) and token.
template <typename T, bool kRes, bool kDL>
__device__ __forceinline__ float queue_weight(const RaceRow<T> &r, const SearchSmem &sm, int e)
{
    const int warp = threadIdx.x >> 5;
    const float t = sv::exp_f32(__fsub_rn(__fmul_rn(sm.ql[warp * kQueue + e], r.invT), r.m));
    float qv = sm.qq[warp * kQueue + e];  // q, or the raw draft logit (draft-logits mode)
    if constexpr (kDL) qv = __fdiv_rn(sv::exp_f32(__fsub_rn(__fmul_rn(qv, r.invT), r.md)), r.Sd);
    return kRes ? __fmaf_rn(-r.S, qv, t) : t;
}

// flush_queue with binary64 clocks and keys (r.f64): *sm.best receives each key rounded down to
// binary32 (a lower bound, used only to prune), and each warp's exact best (the largest binary64
// key, lowest token on equal keys) goes to wbk / wbv.
template <typename T, bool kRes, bool kDL>
__device__ void flush_queue_f64(const RaceRow<T> &r, const SearchSmem &sm, int n)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int e0 = 0; e0 < n; e0 += 32) {
        const int e = e0 + lane;
        unsigned long long p = 0, kb = 0;  // kb: binary64 key bits + 1 (0: no candidate)
        int kv = INT_MAX;
        if (e < n) {
            const uint32_t gsl = sm.qgs[warp * kQueue + e];
            const int g = static_cast<int>(gsl >> 6), slot = static_cast<int>(gsl & 63u);
            const float w = queue_weight<T, kRes, kDL>(r, sm, e);
            if (!kRes || w > 0.0f) {
                const double k64 = key_f64(w, static_cast<uint32_t>(g) + r.g0, slot, sm.ag[g], r.j,
                                           r.ireq, r.k0, r.k1);
                kb = static_cast<unsigned long long>(__double_as_longlong(k64)) + 1ull;
                kv = g * kGroup + slot;
                p = pack_key(__double2float_rd(k64), kv);
            }
        }
        p = warp_max_u64(p);
        if (lane == 0 && p != 0) atomicMax(sm.best, p);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const unsigned long long k2 = __shfl_xor_sync(0xFFFFFFFFu, kb, o);
            const int v2 = __shfl_xor_sync(0xFFFFFFFFu, kv, o);
            if (k2 > kb || (k2 == kb && v2 < kv)) {
                kb = k2;
                kv = v2;
            }
        }
        if (lane == 0 && (kb > sm.wbk[warp] || (kb == sm.wbk[warp] && kb != 0 && kv < sm.wbv[warp]))) {
            sm.wbk[warp] = kb;
            sm.wbv[warp] = kv;
        }
    }
    __syncwarp();
}

// Empty the warp's candidate queue (n entries): one token per lane, its exact weight, its race
// clock and its key, merged into *sm.best. Entry: group g, slot s, raw logit, q entry.
// Slot s = v & 63 of group g: its clock is E_g for the head's slot a, else fl(E_g + (-log U_s)),
// U_s from word s & 3 of slot call s / 4 (tag kClockHead + 1 + s / 4). Binary64 races take
// flush_queue_f64.
template <typename T, bool kRes, bool kDL>
__device__ void flush_queue(const RaceRow<T> &r, const SearchSmem &sm, int n)
{
    __syncwarp();
    if (r.f64) {
        flush_queue_f64<T, kRes, kDL>(r, sm, n);
        return;
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int e0 = 0; e0 < n; e0 += 32) {
        const int e = e0 + lane;
        unsigned long long p = 0;
        if (e < n) {
            const uint32_t gsl = sm.qgs[warp * kQueue + e];
            const int g = static_cast<int>(gsl >> 6), slot = static_cast<int>(gsl & 63u);
            const float w = queue_weight<T, kRes, kDL>(r, sm, e);
            if (!kRes || w > 0.0f) {
                const uint32_t wh = sm.ew[g];
                const float E = group_emin_word(wh);
                float Ev = E;
                if (slot != sm.ag[g]) {
                    const sv::Philox4 sl = sv::philox4x32_10(
                        static_cast<uint32_t>(g) + r.g0, r.j, r.ireq,
                        sv::kClockHead + 1u + static_cast<uint32_t>(slot >> 2), r.k0, r.k1);
                    const uint32_t ws = (slot & 2) ? ((slot & 1) ? sl.w : sl.z) : ((slot & 1) ? sl.y : sl.x);
                    Ev = __fadd_rn(E, -sv::log_f32(sv::uniform_from_word(ws)));
                }
                p = pack_key(__fdiv_rn(w, Ev), g * kGroup + slot);
            }
        }
        p = warp_max_u64(p);
        if (lane == 0 && p != 0) atomicMax(sm.best, p);
    }
    __syncwarp();
}

// Stage 1 of up to B groups by one warp (two adjacent tokens per lane and group; gs[k] < 0: no
// group): every token whose key can still reach the best found so far joins the warp's queue,
// by an upper bound from the hardware ex2 / lg2 / rcp with margins (key_v <= w_v / E_g; weights
// at most exp(x - m), and the residual's fma is monotone in it). The queue is emptied through
// flush_queue whenever it holds 32 tokens; qn is its length. In draft-logits mode q_v is bounded
// from below the same way (hardware ex2 and a reciprocal of S_d, with margins). kOnePerLane: of
// its two tokens a lane queues only the one with the larger bound (a first threshold from at most
// 32 exact keys; the group's other tokens are left to a later evaluation).
template <typename T, bool kRes, bool kDL, bool kPen, int B, bool kOnePerLane = false>
__device__ __forceinline__ void eval_groups(const RaceRow<T> &r, const int (&gs)[B], const SearchSmem &sm,
                                            int &qn)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float l[B][2], qv[B][2];
#pragma unroll
    for (int k = 0; k < B; ++k) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int v = gs[k] * kGroup + 2 * lane + h;
            const bool in = gs[k] >= 0 && v < r.V;
            const float raw = in ? Elem<T>::at(r.rp, v) : -kInf;
            l[k][h] = kPen && in ? pen_apply(r.pr, raw, v) : raw;
            qv[k][h] = 0.0f;
            if constexpr (kRes && kDL) qv[k][h] = in ? Elem<T>::at(r.dlrow, v) : 0.0f;
            else if constexpr (kRes) qv[k][h] = in ? sv_ldg(r.qrow + v) : 0.0f;
        }
    }
    const float inv_sd = kDL ? __frcp_rz(r.Sd) * (1.0f - 0x1p-12f) : 0.0f;  // <= 1 / S_d
    const unsigned long long cur = ld_best(sm.best);
    const unsigned thr = static_cast<unsigned>(cur >> 32);
#pragma unroll
    for (int k = 0; k < B; ++k) {
        const int g = gs[k];
        if (g < 0) continue;
        const float inv = inv_emin_bound(head_uniform_ub(sm.ew[g], r.f64));
        bool tk[2];
        float kbv[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int v = g * kGroup + 2 * lane + h;
            const float xv = __fmul_rn(l[k][h], r.invT);
            const float y = __fsub_rn(xv, r.m);
            const float t_ub = sv::ex2_approx(y * kLog2e) * (1.0f + 0x1p-12f);
            float q_lb = qv[k][h];
            if constexpr (kDL) {
                const float yd = __fsub_rn(__fmul_rn(qv[k][h], r.invT), r.md);
                // exp_f32 is 0 below -87: the bound must be too
                q_lb = yd >= -87.0f ? sv::ex2_approx(yd * kLog2e) * (1.0f - 0x1p-12f) * inv_sd : 0.0f;
            }
            const float w_ub = kRes ? __fmaf_rn(-r.S, q_lb, t_ub) : t_ub;
            bool take = v < r.V && (kRes ? w_ub > 0.0f : v != r.excl) && xv >= r.tau;
            kbv[h] = w_ub * inv * (1.0f + 0x1p-12f);
            if (take && cur != 0) take = !(kbv[h] == kbv[h]) || key_enc(kbv[h]) >= thr;  // NaN kept
            tk[h] = take;
        }
        if constexpr (kOnePerLane) {
            if (tk[0] && tk[1]) {
                if (kbv[1] > kbv[0]) tk[0] = false;
                else tk[1] = false;
            }
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int v = g * kGroup + 2 * lane + h;
            const bool take = tk[h];
            const unsigned msk = __ballot_sync(0xFFFFFFFFu, take);
            if (take) {
                const int pos = warp * kQueue + qn + __popc(msk & ((1u << lane) - 1u));
                sm.qgs[pos] = (static_cast<uint32_t>(g) << 6) | static_cast<uint32_t>(v & 63);
                sm.ql[pos] = l[k][h];
                sm.qq[pos] = qv[k][h];
            }
            qn += __popc(msk);
        }
        if (qn >= 32) {
            flush_queue<T, kRes, kDL>(r, sm, qn);
            qn = 0;
        }
    }
}

// Bin of a key bound (encoded kb) among kBins log-spaced bins from log2(top) down to bottom
// (bin 0 = the largest bounds; NaN / inf and anything lower go to the last bin). The bins only
// order the evaluation: any placement is correct.
__device__ __forceinline__ int bound_bin(unsigned kb, float top, float inv_w)
{
    const float t = (top - __log2f(key_dec(kb))) * inv_w;
    return t < static_cast<float>(kBins - 1) ? (t > 0.0f ? static_cast<int>(t) : 0) : kBins - 1;
}

// Best-first race over one row by the whole CTA. Returns the packed winner (key, ~v), 0 when no
// token is a candidate (binary64 races: the winner's key rounded down to binary32). lm must
// hold the row's line maxima (it is overwritten).
template <typename T, bool kRes, bool kDL, bool kPen>
__device__ unsigned long long race_search(const RaceRow<T> &r, const RowLines &rl,
                                          const SearchSmem &sm)
{
    constexpr int B = 4;  // groups per warp and step
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned long long mine = group_bounds<T>(r, rl, sm);
    if (tid == 0) {
        *sm.best = 0;
        *sm.cnt = 0;
        *sm.top = 0u;
    }
    if (lane == 0) {
        sm.wbk[warp] = 0ull;
        sm.wbv[warp] = INT_MAX;
    }
    if (tid < kBins) {
        sm.bin_n[tid] = 0;
        sm.bin_max[tid] = 0u;
    }
    __syncthreads();  // bounds complete: lm is free from here on (buf reuses it)
    // round 1: every warp evaluates one token per lane of its own best-bounded group
    const unsigned long long wb = warp_max_u64(mine);
    if (lane == 0) atomicMax(sm.top, static_cast<unsigned>(wb >> 32));
    if (wb != 0) {  // (the group stays a candidate: half of it is evaluated here)
        const int gs[1] = {static_cast<int>(~static_cast<unsigned>(wb))};
        int qn = 0;
        eval_groups<T, kRes, kDL, kPen, 1, true>(r, gs, sm, qn);
        flush_queue<T, kRes, kDL>(r, sm, qn);
    }
    __syncthreads();
    // round 2: every group whose bound reaches the best key found so far, best bound first:
    // the candidates are listed with their bin (log-spaced between the largest bound and the
    // best key), counted per bin, then placed in bin order
    const unsigned long long best1 = *sm.best;
    const unsigned thr1 = static_cast<unsigned>(best1 >> 32);
    const float top = __log2f(key_dec(*sm.top));
    const float bottom = fmaxf(best1 != 0 ? __log2f(key_dec(thr1)) : -kInf, top - 48.0f);
    const float inv_w = top - bottom > 0.0f ? kBins / (top - bottom) : 0.0f;
    for (int g0 = 0; g0 < r.G; g0 += kThreads) {
        const int g = g0 + tid;
        unsigned kb = 0;
        bool take = false;
        if (g < r.G) {
            const float b = sm.pb[g];
            if (b == b) {
                kb = key_enc(key_bound(b));
                take = best1 == 0 || kb >= thr1;
            }
        }
        int bin = 0;
        if (take) {
            bin = bound_bin(kb, top, inv_w);
            atomicAdd(&sm.bin_n[bin], 1);
            atomicMax(&sm.bin_max[bin], kb);
        }
        const unsigned msk = __ballot_sync(0xFFFFFFFFu, take);
        int pos = 0;
        if (lane == 0 && msk) pos = atomicAdd(sm.cnt, __popc(msk));
        pos = __shfl_sync(0xFFFFFFFFu, pos, 0) + __popc(msk & ((1u << lane) - 1u));
        if (take)
            sm.buf[pos] = (static_cast<unsigned long long>(kb) << 32) |
                          (static_cast<unsigned>(bin) << 24) | static_cast<unsigned>(g);
    }
    __syncthreads();
    const int cnt = *sm.cnt;
    if (tid < 32) {  // exclusive prefix of the bin counts (kBins == 32): the bins' cursors
        const int nb = sm.bin_n[tid];
        int x = nb;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (tid >= o) x += y;
        }
        sm.bin_n[tid] = x - nb;
    }
    __syncthreads();
    for (int e = tid; e < cnt; e += kThreads) {
        const unsigned long long ent = sm.buf[e];
        sm.tmp[atomicAdd(&sm.bin_n[(ent >> 24) & 0xFFu], 1)] = ent;
    }
    __syncthreads();
    int qn = 0;
    for (int e0 = warp * B; e0 < cnt; e0 += kWarps * B) {
        const unsigned long long cur = ld_best(sm.best);
        const unsigned thr = static_cast<unsigned>(cur >> 32);
        int gs[B];
        bool done = false;
#pragma unroll
        for (int k = 0; k < B; ++k) {
            gs[k] = -1;
            const int e = e0 + k;
            if (e < cnt && !done) {
                const unsigned long long ent = sm.tmp[e];
                const int bin = static_cast<int>((ent >> 24) & 0xFFu);
                if (cur != 0 && sm.bin_max[bin] < thr) {
                    done = true;  // this bin and every later one lie below the best key
                } else if (cur == 0 || static_cast<unsigned>(ent >> 32) >= thr) {
                    gs[k] = static_cast<int>(ent & 0x00FFFFFFull);
                }
            }
        }
        eval_groups<T, kRes, kDL, kPen, B>(r, gs, sm, qn);
        if (qn > 0) {  // keys now: the best key prunes the next groups
            flush_queue<T, kRes, kDL>(r, sm, qn);
            qn = 0;
        }
        if (done) break;
    }
    __syncthreads();
    if (r.f64) {  // the exact winner over the warps' binary64 bests
        unsigned long long kb = 0ull;
        int kv = INT_MAX;
        for (int w = 0; w < kWarps; ++w)
            if (sm.wbk[w] > kb || (sm.wbk[w] == kb && kb != 0ull && sm.wbv[w] < kv)) {
                kb = sm.wbk[w];
                kv = sm.wbv[w];
            }
        __syncthreads();  // every thread has read wbk / wbv before a next race resets them
        return kb ? pack_key(__double2float_rd(__longlong_as_double(static_cast<long long>(kb - 1ull))), kv)
                  : 0ull;
    }
    return *sm.best;
}

// The statistics of one row from its partials, by one warp: (max raw logit, sum of
// 2^((l - L) c), lowest argmax); every warp of every segment wrote one partial, in segment order.
__device__ __forceinline__ void combine_row(const StatPart *__restrict__ part, long long row, int V,
                                            int maxseg, int base_off, const Divisor &chunk, float c,
                                            float &L, float &s, int &idx)
{
    const int lane = threadIdx.x & 31;
    const long long rbase = row * V;
    const int nseg = static_cast<int>(div_floor(base_off + rbase + V - 1, chunk) -
                                      div_floor(base_off + rbase, chunk)) + 1;
    L = -kInf;
    s = 0.0f;
    idx = INT_MAX;
    for (int k = lane; k < nseg * kWarps; k += 32) {
        const float4 raw = sv_ldg(reinterpret_cast<const float4 *>(part) +
                                 static_cast<size_t>(row) * maxseg * kWarps + k);
        combine_stat(L, s, idx, raw.x, raw.y, __float_as_int(raw.z), c);
    }
    warp_reduce_stat(L, s, idx, c);
}

// The row's lowest index of its maximum L from the combined candidate `cand` (argmax_candidate;
// 0 for none), by the whole warp: a pair is read once, an element per lane, and the lowest lane
// holding L is the index.
template <typename T>
__device__ __forceinline__ int resolve_argmax(const T *__restrict__ rp, int cand, float L)
{
    if (cand == INT_MAX) return 0;
    const int a = cand >> 1;
    if (!(cand & 1)) return a;
    constexpr int kPE = kPairBytes / static_cast<int>(sizeof(T));
    const int lane = threadIdx.x & 31;
    const bool hit = lane < kPE && Elem<T>::at(rp, a + lane) == L;
    const unsigned b = __ballot_sync(0xFFFFFFFFu, hit);
    return b ? a + __ffs(b) - 1 : a;  // (a pair always holds its maximum)
}

// ---------------------------------------------------------------------------------------
// 3. sampling constraints: top-k / top-p of one row ([spec-notes] 8.2
//    apply_sampling_constraints; [mini-sglang] "how tokens are sampled")
// ---------------------------------------------------------------------------------------
// The kept tokens of a constrained row are {x_v >= tau}:
//   top-k: tau_k = the k-th largest x (ties at it are kept), for 1 <= k < V;
//   top-p: among those, every token whose strictly larger tokens hold less than P * Z of the
//          mass t_v = exp(x_v - m), Z the mass of the top-k set, for P < 1 (at least 1e-6).
// One CTA per row finds tau without sorting the row: a histogram of counts (top-k) or masses
// (top-p) over 256 bins of 1/8 nat below the row maximum, one atomic per token into its warp's
// copy (one pass over the row); then the bin where the k-th token or the P * Z mass falls is
// collected into shared memory (a second pass, from L2) and refined there on the
// order-preserving integer key of x, 8 bits per level, down to a single value (a group of equal
// values is kept or dropped as a whole); a bin too large to collect is refined over the row
// first. Masses come from the hardware ex2, summed in fp32.
constexpr int kSelBins1 = 2048;         // level 1: counts in bins of 1/64 nat below the maximum
constexpr float kSelBinsPerNat = 64.0f;
constexpr int kSelBins = 256;           // the finer levels: 8 key bits each
constexpr int kSelPool = 2048;          // tokens refined in shared memory
static_assert(kSelBins == kThreads && kSelBins1 % kThreads == 0, "bins per thread");

struct SelectParams {
    RequestTable rq;
    PenTable pen;
    const int32_t *draft_ids;
    const int32_t *top_k;
    const float *top_p;
    const StatPart *part;
    int V, maxseg, base_off;
    Divisor chunk;
    float *sel_tau;  // [rows] threshold of each constrained row
    float *sel_S;    // [rows] its kept mass: the normaliser of p'
    int lmx_cap;     // line maxima the dynamic shared memory holds after the pools
    unsigned *flags; // the call's error word pair
};

// Does request i sample under constraints? (k, P as given; greedy requests never do.)
__device__ __forceinline__ bool sel_active(const int32_t *top_k, const float *top_p, int i, int V,
                                           bool greedy, int &k, float &P)
{
    k = top_k ? sv_ldg(top_k + i) : 0;
    P = top_p ? sv_ldg(top_p + i) : 1.0f;
    return !greedy && ((k >= 1 && k < V) || P < 1.0f);
}

// Integer key in the order of the values; -0 takes the key of +0, so that equal values have
// equal keys.
__device__ __forceinline__ uint32_t ord_key(float x)
{
    const uint32_t u = x == 0.0f ? 0u : __float_as_uint(x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
// Level-1 bin: 0 holds the values less than 1/64 nat below m, the last everything further down
// than 2047/64 nats. u = (m - x) 64 is clamped to [0, 2047] (NaN: the last bin) and truncated by
// a round-toward-zero add into the significand of 2^23 (full-rate float and integer operations
// instead of a conversion).
__device__ __forceinline__ int sel_bin1(float x, float m)
{
    const float u = fmaxf(fminf(__fmul_rn(__fsub_rn(m, x), kSelBinsPerNat),
                                static_cast<float>(kSelBins1 - 1)), 0.0f);
    return __float_as_int(__fadd_rz(u, 8388608.0f)) - 0x4B000000;
}
// A token's mass exp(x - m), by the hardware ex2.
__device__ __forceinline__ float sel_mass(float x, float m)
{
    return sv::ex2_approx(__fmul_rn(__fsub_rn(x, m), kLog2e));
}

// Dynamic shared memory of the select kernel (40 KB: four CTAs per SM at 64 registers):
// [kWarps][kSelBins] per-warp counts or masses (float bits) of the finer levels, the level-1
// counts [kSel1Copies][kSelBins1] (a copy per four warps), then two pools of kSelPool tokens.
constexpr int kSel1Copies = kWarps / 4;
extern __shared__ __align__(16) unsigned char sv_sel_dyn[];

struct SelSmem {
    __device__ __forceinline__ uint32_t *hist() const { return reinterpret_cast<uint32_t *>(sv_sel_dyn); }
    __device__ __forceinline__ uint32_t *cnt1() const { return hist() + kWarps * kSelBins; }
    __device__ __forceinline__ float *pool_a() const
    {
        return reinterpret_cast<float *>(cnt1() + kSel1Copies * kSelBins1);
    }
    // a level-1 bin's count over the copies
    __device__ __forceinline__ uint32_t count1(int b) const
    {
        uint32_t c = 0u;
        for (int w = 0; w < kSel1Copies; ++w) c += cnt1()[w * kSelBins1 + b];
        return c;
    }
    __device__ __forceinline__ float *pool_b() const { return pool_a() + kSelPool; }
    // the row's line maxima in x units (rows read by lines only), after the pools, then the
    // warps' vector queues (kWarps x kSelQueue) after lmx_cap of them
    __device__ __forceinline__ float *lmx() const { return pool_b() + kSelPool; }
    __device__ __forceinline__ uint32_t *wq(int lmx_cap) const
    {
        return reinterpret_cast<uint32_t *>(lmx() + lmx_cap);
    }
    uint32_t wc[kWarps];
    float wm[kWarps];
    uint32_t kmin, kmax, n;
    int cross;
    float fsum;
    uint32_t cabove;
    float mabove;
};

// Every element of a row once, as x = processed logit * (1 / T), with its token index: 16-byte
// loads over the aligned body, four in flight per thread (with a penalty, each with its counts,
// 16-byte loads where the counts row is so aligned). The rounds are uniform over the warp (a
// lane past the end takes part without an element), so that the earlier drafts (lane k holding
// the k-th, k < 32) are tested against the warp's window of tokens by one ballot per vector
// round; only a window that holds one adds them token by token.
template <typename T, bool kPen, typename F>
__device__ __forceinline__ void sel_for_row(const T *__restrict__ rp, int V, float invT,
                                            const PenRow &pr, F &&f)
{
    constexpr int kEV = 16 / static_cast<int>(sizeof(T));
    constexpr int kIn = 4;
    constexpr int kCV = kPen ? kEV / 4 : 1;  // 16-byte count vectors per logit vector
    const int head = min(V, static_cast<int>(((16u - (reinterpret_cast<uintptr_t>(rp) & 15u)) & 15u) / sizeof(T)));
    auto proc = [&](float l, int v) { return __fmul_rn(kPen ? pen_apply(pr, l, v) : l, invT); };
    for (int v = threadIdx.x; v < head; v += kThreads) f(proc(Elem<T>::at(rp, v), v), v);
    const int nvec = (V - head) / kEV;
    const char *base = reinterpret_cast<const char *>(rp + head);
    const int lane = threadIdx.x & 31;
    const bool pen = kPen && pr.f != 0.0f;
    const bool al = pen && (reinterpret_cast<uintptr_t>(pr.cnt + head) & 15u) == 0u;
    const int pv = pen && lane < pr.nprev ? sv_ldg(pr.prev + lane) : -1;
    for (int u0 = threadIdx.x; (u0 & ~31) < nvec; u0 += kIn * kThreads) {
        uint4 w[kIn];
        int4 cv[kIn][kCV];
        bool scan[kIn];
#pragma unroll
        for (int q = 0; q < kIn; ++q) {
            const int u = u0 + q * kThreads;
            w[q] = u < nvec ? ldg_v4(base + static_cast<size_t>(u) * 16) : make_uint4(0, 0, 0, 0);
            if constexpr (kPen) {
#pragma unroll
                for (int g = 0; g < kCV; ++g)
                    cv[q][g] = al && u < nvec
                                   ? sv_ldg(reinterpret_cast<const int4 *>(pr.cnt + head + u * kEV) + g)
                                   : make_int4(0, 0, 0, 0);
                const int wlo = head + ((u0 & ~31) + q * kThreads) * kEV;  // the warp's window
                scan[q] = pen && (pr.nprev > 32 ||
                                  __ballot_sync(0xFFFFFFFFu, static_cast<unsigned>(pv - wlo) <
                                                                 static_cast<unsigned>(32 * kEV)) != 0u);
            }
        }
#pragma unroll
        for (int q = 0; q < kIn; ++q) {
            const int u = u0 + q * kThreads;
            if (u >= nvec) break;
            const uint32_t ws[4] = {w[q].x, w[q].y, w[q].z, w[q].w};
            const int v0 = head + u * kEV;
            int cnt[kEV];
            if constexpr (kPen) {
                if (al) {
#pragma unroll
                    for (int g = 0; g < kCV; ++g) {
                        cnt[4 * g] = cv[q][g].x;
                        cnt[4 * g + 1] = cv[q][g].y;
                        cnt[4 * g + 2] = cv[q][g].z;
                        cnt[4 * g + 3] = cv[q][g].w;
                    }
                } else {
#pragma unroll
                    for (int e = 0; e < kEV; ++e) cnt[e] = pen ? sv_ldg(pr.cnt + v0 + e) : 0;
                }
                if (scan[q])
                    for (int g = 0; g < pr.nprev; ++g) {
                        const int d = sv_ldg(pr.prev + g) - v0;
#pragma unroll
                        for (int e = 0; e < kEV; ++e) cnt[e] += d == e;
                    }
            }
#pragma unroll
            for (int e = 0; e < kEV; ++e) {
                float l;
                if constexpr (sizeof(T) == 2)
                    l = __uint_as_float((e & 1) ? (ws[e >> 1] & 0xFFFF0000u) : (ws[e >> 1] << 16));
                else
                    l = __uint_as_float(ws[e]);
                const int v = v0 + e;
                if constexpr (kPen) {
                    const float y = cnt[e] == 0 ? l : __fmaf_rn(-pr.f, __int2float_rn(cnt[e]), l);
                    f(__fmul_rn(y, invT), v);
                } else {
                    f(__fmul_rn(l, invT), v);
                }
            }
        }
    }
    for (int v = head + nvec * kEV + threadIdx.x; v < V; v += kThreads)
        f(proc(Elem<T>::at(rp, v), v), v);
}

constexpr size_t kSelDynSmem =
    (static_cast<size_t>(kWarps) * kSelBins + static_cast<size_t>(kSel1Copies) * kSelBins1 +
     2 * kSelPool) * 4;

// Every element of a row whose x = fl(l * invT) can reach xmin, as (x, token), reading only the
// 64-element lines whose largest x (lmx[k], from the statistics pass's line maxima) reaches
// xmin and, inside them, only the 16-byte vectors whose largest x does: x is monotone in l, so
// a vector's largest x is fl(vector max * invT) and a line's is lmx. The vectors that pass are
// queued per warp (their index in wq, their data in wqd: kSelQueue entries per warp, in shared
// memory) and processed 32 at a time, one per lane, so that the few that pass do not each hold
// a mostly idle warp through their elements. The loads of a step are issued before the step
// before it is processed (two register buffers in rotation). Elements below xmin may still be
// passed (callers test x); the partial first and last lines of the row go element by element.
// f takes no warp-wide step.
constexpr int kSelQueue = 64;
// Vectors per lane and load buffer of the selection's row passes: two in the count pass, one in
// the passes that hand tokens to a callback (their loop bodies are larger; one vector measured
// 350 against 405 us for top-p 0.9 on the 256-request bf16 workload, the count pass better at two).
constexpr int kSelUnrollCount = 2;
constexpr int kSelUnrollRead = 1;
static_assert(kWarps * kSelQueue * 16 == kSelPool * 4, "the queued vectors' data fills pool_b");

template <typename T, int kSelUnroll>
struct RowSteps {  // the whole lines of a row, in steps of kWarps * kLPW * kSelUnroll lines
    static constexpr int kEV = 16 / static_cast<int>(sizeof(T));  // elements per vector
    static constexpr int kVPL = kGroup / kEV;                      // vectors per line
    static constexpr int kLPW = 32 / kVPL;                         // lines per warp and unit
    static constexpr int kStep = kWarps * kLPW * kSelUnroll;       // lines per CTA step
    const char *base;  // line kf's first byte
    int nfull, kf, tok0, sub, lsub;
    __device__ __forceinline__ RowSteps(const T *rp, const RowLines &rl)
    {
        nfull = max(0, rl.kl - rl.kf + 1);
        kf = rl.kf;
        tok0 = static_cast<int>((rl.L0 + rl.kf) * kGroup - rl.P0);
        base = reinterpret_cast<const char *>(rp + tok0);
        sub = (threadIdx.x & 31) % kVPL;
        lsub = (threadIdx.x & 31) / kVPL;
    }
    // line of unit u of the step starting at lb (lb uniform over the warp)
    __device__ __forceinline__ int line(int lb, int u) const { return lb + u * kWarps * kLPW + lsub; }
    // issue the loads of the step at lb: vectors of lines whose maximum reaches xmin
    __device__ __forceinline__ void load(int lb, const float *lmx, float xmin, uint4 (&w)[kSelUnroll],
                                         bool (&act)[kSelUnroll]) const
    {
#pragma unroll
        for (int u = 0; u < kSelUnroll; ++u) {
            const int ln = line(lb, u);
            act[u] = ln < nfull && lmx[kf + ln] >= xmin;
            w[u] = act[u] ? ldg_v4(base + (static_cast<size_t>(ln) * kVPL + sub) * 16)
                          : make_uint4(0u, 0u, 0u, 0u);
        }
    }
};

// The partial first (warp 0) and last (warp 1) lines of a row, element by element.
template <typename T, typename F>
__device__ __forceinline__ void sel_partial_lines(const T *__restrict__ rp, int V, float invT,
                                                  const RowLines &rl, const float *lmx, float xmin,
                                                  F &&f)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int k = -1;
    if (warp == 0 && rl.kf == 1) k = 0;
    if (warp == 1 && rl.kl == rl.nl - 2 && (rl.nl > 1 || rl.kf == 0)) k = rl.nl - 1;
    if (k >= 0 && lmx[k] >= xmin) {
        const long long p = (rl.L0 + k) * kGroup;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const long long v = p + h * 32 + lane - rl.P0;
            if (v >= 0 && v < V) f(__fmul_rn(Elem<T>::at(rp, static_cast<size_t>(v)), invT), static_cast<int>(v));
        }
    }
}

template <typename T, typename F>
__device__ __forceinline__ void sel_for_row_lines(const T *__restrict__ rp, int V, float invT,
                                                  const RowLines &rl, const float *lmx, float xmin,
                                                  uint32_t *wq, uint4 *wqd, F &&f)
{
    constexpr int kSelUnroll = kSelUnrollRead;
    using RS = RowSteps<T, kSelUnroll>;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    sel_partial_lines<T>(rp, V, invT, rl, lmx, xmin, [&](float x, int v) {
        if (x >= xmin) f(x, v);
    });
    const RS rs(rp, rl);
    uint32_t *q = wq + warp * kSelQueue;
    uint4 *qd = wqd + warp * kSelQueue;
    int qn = 0;
    auto elems = [&](const uint4 &w, uint32_t vi) {  // the elements of vector vi (from line kf)
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
        const int v0 = rs.tok0 + static_cast<int>(vi) * RS::kEV;
#pragma unroll
        for (int e = 0; e < RS::kEV; ++e) {
            float l;
            if constexpr (sizeof(T) == 2)
                l = __uint_as_float((e & 1) ? (ws[e >> 1] & 0xFFFF0000u) : (ws[e >> 1] << 16));
            else
                l = __uint_as_float(ws[e]);
            const float x = __fmul_rn(l, invT);
            if (x >= xmin) f(x, v0 + e);
        }
    };
    // queue the vectors of a loaded step that can reach xmin; process 32 of them whenever 32 wait
    auto step = [&](int lb, const uint4 (&w)[kSelUnroll], const bool (&act)[kSelUnroll]) {
#pragma unroll
        for (int u = 0; u < kSelUnroll; ++u) {
            const bool pass = act[u] && __fmul_rn(VecMax<T>::value(VecMax<T>::of(w[u])), invT) >= xmin;
            const unsigned msk = __ballot_sync(0xFFFFFFFFu, pass);
            if (pass) {
                const int at = qn + __popc(msk & ((1u << lane) - 1u));
                q[at] = static_cast<uint32_t>(rs.line(lb, u) * RS::kVPL + rs.sub);
                qd[at] = w[u];
            }
            qn += __popc(msk);
            if (qn >= 32) {  // the last 32 queued vectors, one per lane
                __syncwarp();
                elems(qd[qn - 32 + lane], q[qn - 32 + lane]);
                qn -= 32;
                __syncwarp();
            }
        }
    };
    uint4 wa[kSelUnroll], wb[kSelUnroll];
    bool aa[kSelUnroll], ab[kSelUnroll];
    int lb = warp * RS::kLPW;  // uniform over the warp
    rs.load(lb, lmx, xmin, wa, aa);
    while (lb < rs.nfull) {
        rs.load(lb + RS::kStep, lmx, xmin, wb, ab);
        step(lb, wa, aa);
        lb += RS::kStep;
        if (lb >= rs.nfull) break;
        rs.load(lb + RS::kStep, lmx, xmin, wa, aa);
        step(lb, wb, ab);
        lb += RS::kStep;
    }
    __syncwarp();
    if (lane < qn) elems(qd[lane], q[lane]);
    __syncwarp();
}

// Level-1 counts (into `cnt`, one shared atomic per token) of a row's tokens with x >= xmin, read
// as sel_for_row_lines reads them (lines and vectors that cannot reach xmin are skipped, loads a
// step ahead), with the per-token work cut down: x = fl(l * invT) and the bin's fl(m - x) * 64
// (the value sel_bin1 clamps, so both passes bin every token alike) two tokens per packed
// binary32 instruction. Vectors are processed where they were loaded (almost all of them are,
// in this pass).
template <typename T>
__device__ __forceinline__ void sel_count_lines(const T *__restrict__ rp, int V, float invT, float m,
                                                const RowLines &rl, const float *lmx, float xmin,
                                                uint32_t *cnt)
{
    constexpr int kSelUnroll = kSelUnrollCount;
    using RS = RowSteps<T, kSelUnroll>;
    sel_partial_lines<T>(rp, V, invT, rl, lmx, xmin, [&](float x, int) {
        if (x >= xmin) atomicAdd(cnt + sel_bin1(x, m), 1u);
    });
    const RS rs(rp, rl);
    const int warp = threadIdx.x >> 5;
    const unsigned long long ninv2 = f2_pack(-invT, -invT), m2 = f2_pack(m, m);
    const unsigned long long s2 = f2_pack(kSelBinsPerNat, kSelBinsPerNat);
    const float nxmin = -xmin;
    auto step = [&](const uint4 (&w)[kSelUnroll], const bool (&act)[kSelUnroll]) {
#pragma unroll
        for (int u = 0; u < kSelUnroll; ++u) {
            if (!act[u]) continue;
            if (!(__fmul_rn(VecMax<T>::value(VecMax<T>::of(w[u])), invT) >= xmin)) continue;
            const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
            for (int q = 0; q < RS::kEV / 2; ++q) {
                unsigned long long l2;
                if constexpr (sizeof(T) == 2)
                    l2 = f2_pack(__uint_as_float(ws[q] << 16), __uint_as_float(ws[q] & 0xFFFF0000u));
                else
                    l2 = f2_pack(__uint_as_float(ws[2 * q]), __uint_as_float(ws[2 * q + 1]));
                const unsigned long long nx2 = f2_mul(l2, ninv2);           // -x = fl(l * -invT)
                const unsigned long long u2 = f2_mul(f2_add(m2, nx2), s2);  // fl(m - x) * 64
                float nx0, nx1, u0, u1;
                f2_unpack(nx2, nx0, nx1);
                f2_unpack(u2, u0, u1);
                // x >= xmin (false for NaN); the bin as sel_bin1 clamps and truncates it
                if (nx0 <= nxmin)
                    atomicAdd(cnt + (__float_as_int(__fadd_rz(fmaxf(fminf(u0, static_cast<float>(kSelBins1 - 1)), 0.0f), 8388608.0f)) - 0x4B000000), 1u);
                if (nx1 <= nxmin)
                    atomicAdd(cnt + (__float_as_int(__fadd_rz(fmaxf(fminf(u1, static_cast<float>(kSelBins1 - 1)), 0.0f), 8388608.0f)) - 0x4B000000), 1u);
            }
        }
    };
    uint4 wa[kSelUnroll], wb[kSelUnroll];
    bool aa[kSelUnroll], ab[kSelUnroll];
    int lb = warp * RS::kLPW;
    rs.load(lb, lmx, xmin, wa, aa);
    while (lb < rs.nfull) {
        rs.load(lb + RS::kStep, lmx, xmin, wb, ab);
        step(wa, aa);
        lb += RS::kStep;
        if (lb >= rs.nfull) break;
        rs.load(lb + RS::kStep, lmx, xmin, wa, aa);
        step(wb, ab);
        lb += RS::kStep;
    }
}

// The smallest x that can lie in level-1 bins 0 .. b (one bin of slack against the rounding of
// sel_bin1); -inf for the last bins, which take everything below.
__device__ __forceinline__ float sel_bin1_floor(int b, float m)
{
    return b < kSelBins1 - 2 ? __fsub_rn(m, static_cast<float>(b + 2) * (1.0f / kSelBinsPerNat)) : -kInf;
}

__device__ __forceinline__ void sel_clear(SelSmem &sm, int nbins)
{
    for (int k = threadIdx.x; k < kWarps * nbins; k += kThreads) sm.hist()[k] = 0u;
}
__device__ __forceinline__ void sel_add(SelSmem &sm, int mode, int b, float t)
{
    uint32_t *cell = sm.hist() + (threadIdx.x >> 5) * kSelBins + b;
    if (mode == 0) atomicAdd(cell, 1u);
    else atomicAdd(reinterpret_cast<float *>(cell), t);
}

// Sum of a float over the CTA (every thread gets it).
__device__ __forceinline__ float sel_block_sum(SelSmem &sm, float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) sm.wm[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.0f;
    for (int w = 0; w < kWarps; ++w) t += sm.wm[w];
    __syncthreads();
    return t;
}

// After the per-warp histograms over nbins bins are complete (bin 0 holds the largest values):
// the crossing bin. mode 0 (counts): the first bin where ca + count >= k; mode 1 (masses): the
// first bin where ma + mass >= target, or the last non-empty bin if rounding leaves the total
// short. Adds the count (mode 0) or mass (mode 1) strictly above the crossing bin to ca / ma.
// Thread t scans bins [t * per, (t + 1) * per); the prefix of bin b is formed in one fixed
// order, so the excluded sum of a bin is exactly the included sum of the one before.
__device__ int sel_cross(SelSmem &sm, int nbins, int mode, uint32_t k, float target, uint32_t &ca,
                         float &ma)
{
    const int per = nbins / kThreads, b0 = threadIdx.x * per;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // nbins == kSelBins1: the level-1 counts; else the per-warp copies of the finer levels
    auto bin_c = [&](int b) {
        if (nbins == kSelBins1) return sm.count1(b);
        uint32_t c = 0u;
        for (int w = 0; w < kWarps; ++w) c += sm.hist()[w * kSelBins + b];
        return c;
    };
    auto bin_m = [&](int b) {
        float m = 0.0f;
        for (int w = 0; w < kWarps; ++w) m += __uint_as_float(sm.hist()[w * kSelBins + b]);
        return m;
    };
    uint32_t tc = 0u;
    float tm = 0.0f;
    for (int q = 0; q < per; ++q) {
        if (mode == 0) tc += bin_c(b0 + q);
        else tm = tm + bin_m(b0 + q);
    }
    uint32_t ci = tc;
    float mi = tm;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t c2 = __shfl_up_sync(0xFFFFFFFFu, ci, o);
        const float m2 = __shfl_up_sync(0xFFFFFFFFu, mi, o);
        if (lane >= o) {
            ci += c2;
            mi = m2 + mi;
        }
    }
    const uint32_t cprev = __shfl_up_sync(0xFFFFFFFFu, ci, 1);
    const float mprev = __shfl_up_sync(0xFFFFFFFFu, mi, 1);
    if (lane == 31) {
        sm.wc[warp] = ci;
        sm.wm[warp] = mi;
    }
    if (threadIdx.x == 0) sm.cross = -1;
    __syncthreads();
    uint32_t coff = 0u;
    float moff = 0.0f;
    for (int w = 0; w < warp; ++w) {
        coff += sm.wc[w];
        moff = moff + sm.wm[w];
    }
    uint32_t cex = ca + coff + (lane ? cprev : 0u);
    float mex = ma + (lane ? moff + mprev : moff);
    int last = -1;
    for (int q = 0; q < per; ++q) {
        const uint32_t c = mode == 0 ? bin_c(b0 + q) : 0u;
        const float mm = mode == 1 ? bin_m(b0 + q) : 0.0f;
        const uint32_t cin = cex + c;
        const float min_ = mex + mm;
        const bool hit = mode == 0 ? (cex < k && cin >= k) : (mex < target && min_ >= target);
        if (hit) {
            sm.cross = b0 + q;
            sm.cabove = cex;
            sm.mabove = mex;
        }
        if (mode == 0 ? c > 0u : mm > 0.0f) last = b0 + q;
        cex = cin;
        mex = min_;
    }
    __syncthreads();
    if (sm.cross < 0) {  // short of the target: the last non-empty bin
        if (threadIdx.x == 0) sm.n = 0u;
        __syncthreads();
        atomicMax(&sm.n, static_cast<uint32_t>(last + 1));
        __syncthreads();
        const int lb = static_cast<int>(sm.n) - 1;
        if (lb >= b0 && lb < b0 + per) {
            uint32_t c2 = ca + coff + (lane ? cprev : 0u);
            float m2 = ma + (lane ? moff + mprev : moff);
            for (int q = b0; q < lb; ++q) {
                if (mode == 0) c2 += bin_c(q);
                else m2 = m2 + bin_m(q);
            }
            sm.cross = lb;
            sm.cabove = c2;
            sm.mabove = m2;
        }
        __syncthreads();
    }
    const int x = max(sm.cross, 0);
    ca = sm.cabove;
    ma = sm.mabove;
    __syncthreads();
    return x;
}

// The level-1 bins where the top-p crossing can lie, from the counts alone: a token of bin b has
// mass in (e^-(b+1)/128, e^-b/128] (the last bin: (0, e^-4095/128]), so the mass up to and
// including bin b lies between the sums of count * lower and count * upper bound (with margins
// for the hardware ex2). Returns the first bin whose upper sum reaches target (no earlier bin can
// hold the crossing) in lo and the first whose lower sum reaches it (no later one can) in hi (the
// last non-empty bin if none does).
__device__ void sel_bounds(SelSmem &sm, float target, int &lo, int &hi)
{
    constexpr int per = kSelBins1 / kThreads;
    const int b0 = threadIdx.x * per, lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t cb[per];  // this thread's bins' counts
    for (int q = 0; q < per; ++q) cb[q] = sm.count1(b0 + q);
    auto bound = [&](int q, bool upper) {
        const int b = b0 + q;
        const float c = static_cast<float>(cb[q]);
        if (!upper && b == kSelBins1 - 1) return 0.0f;
        const float e = sv::ex2_approx(-static_cast<float>(upper ? b : b + 1) * (kLog2e / kSelBinsPerNat));
        return c * e * (upper ? 1.0f + 0x1p-10f : 1.0f - 0x1p-10f);
    };
    float tl = 0.0f, th = 0.0f;
    int last = -1;
    for (int q = 0; q < per; ++q) {
        tl += bound(q, false);
        th += bound(q, true);
        if (cb[q]) last = b0 + q;
    }
    float il = tl, ih = th;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float l2 = __shfl_up_sync(0xFFFFFFFFu, il, o), h2 = __shfl_up_sync(0xFFFFFFFFu, ih, o);
        if (lane >= o) {
            il += l2;
            ih += h2;
        }
    }
    __shared__ float s_wh[kWarps];
    __shared__ int s_lo, s_hi, s_last;
    if (lane == 31) {
        sm.wm[warp] = il;
        s_wh[warp] = ih;
    }
    if (threadIdx.x == 0) {
        s_lo = INT_MAX;
        s_hi = INT_MAX;
        s_last = -1;
    }
    __syncthreads();
    float ol = 0.0f, oh = 0.0f;
    for (int w = 0; w < warp; ++w) {
        ol += sm.wm[w];
        oh += s_wh[w];
    }
    // sums before this thread's first bin (threads differ in rounding; the margins cover it)
    float cl = ol + il - tl, ch = oh + ih - th;
    int flo = INT_MAX, fhi = INT_MAX;
    for (int q = 0; q < per; ++q) {
        cl += bound(q, false);
        ch += bound(q, true);
        if (ch >= target) flo = min(flo, b0 + q);
        if (cl >= target) fhi = min(fhi, b0 + q);
    }
    atomicMin(&s_lo, flo);
    atomicMin(&s_hi, fhi);
    atomicMax(&s_last, last);
    __syncthreads();
    hi = s_hi != INT_MAX ? s_hi : max(s_last, 0);
    lo = min(s_lo != INT_MAX ? s_lo : hi, hi);
    __syncthreads();
}

// Key-level sub-bin of key kv in [klo, khi] with shift sh: 0 holds the largest keys.
__device__ __forceinline__ int sel_sub(uint32_t kv, uint32_t khi, int sh)
{
    return static_cast<int>((khi - kv) >> sh);
}
// The key range of sub-bin sb of [klo, khi] with shift sh.
__device__ __forceinline__ void sel_narrow(uint32_t &klo, uint32_t &khi, int sb, int sh)
{
    const uint32_t nhi = khi - (static_cast<uint32_t>(sb) << sh);
    const uint32_t w = (1u << sh) - 1u;
    klo = nhi - klo >= w ? nhi - w : klo;
    khi = nhi;
}
__device__ __forceinline__ int sel_shift(uint32_t klo, uint32_t khi)
{
    const uint32_t r = khi - klo;
    const int bits = r ? 32 - __clz(r) : 0;
    return bits > 8 ? bits - 8 : 0;
}

// Resolve the crossing among the candidates (each(xmin_hint, f) passes the row's tokens, at least
// those with x >= xmin_hint, to f): the row's tokens with x >= xmin in level-1 bins b1 .. b1hi,
// with ca / ma tokens strictly above them (ca in mode 0, ma in mode 1). The first pass collects
// them into shared memory, counting them and taking their key range (and the mass of the tokens
// in the bins above b1 with x >= xmin, returned in above_mass); only if they do not fit are finer
// levels taken over the row first. Returns x*, the single value where the goal crosses, with
// ca / ma counting / weighing the tokens strictly above x*, inbin_above the mass of the
// candidates strictly above x* (mode 0) and gmass the mass of its group (all tokens equal x*).
template <typename Each>
__device__ float sel_resolve(SelSmem &sm, Each &&each, float m, int b1, int b1hi, float xmin,
                             int mode, uint32_t k, float target, uint32_t &ca, float &ma,
                             float &above_mass, float &inbin_above, float &gmass, bool &gave_up)
{
    // each pass below narrows a window of 32-bit keys at least 128-fold, so a handful of passes
    // always suffice; the limits only turn a defect into a reported error instead of a hang
    constexpr int kMaxRowPasses = 8, kMaxPoolPasses = 8;
    gave_up = false;
    // every token these passes use lies in bins <= b1hi with x >= xmin
    const float hint = fmaxf(xmin, sel_bin1_floor(b1hi, m));
    auto in_set = [&](float x, uint32_t klo, uint32_t khi) {
        const uint32_t kv = ord_key(x);
        const int bx = sel_bin1(x, m);
        return x >= xmin && kv >= klo && kv <= khi && bx >= b1 && bx <= b1hi;
    };
    uint32_t klo = 0u, khi = 0xFFFFFFFFu, n = 0u;
    bool first = true, big = false;
    inbin_above = 0.0f;
    for (int pass = 0;; ++pass) {
        if (pass == kMaxRowPasses) {
            gave_up = true;
            gmass = 0.0f;
            return -kInf;
        }
        if (big && klo < khi) {
            // too many for shared memory: one finer level over the row
            const int sh = sel_shift(klo, khi);
            sel_clear(sm, kSelBins);
            __syncthreads();
            each(hint, [&](float x, int) {
                if (in_set(x, klo, khi)) sel_add(sm, mode, sel_sub(ord_key(x), khi, sh), sel_mass(x, m));
            });
            __syncthreads();
            const int sb = sel_cross(sm, kSelBins, mode, k, target, ca, ma);
            const uint32_t olo = klo, ohi = khi;
            sel_narrow(klo, khi, sb, sh);
            if (mode == 0) {  // the mass of the candidates left above (counts were kept)
                float a = 0.0f;
                const uint32_t nh = khi;
                each(hint, [&](float x, int) {
                    if (in_set(x, olo, ohi) && ord_key(x) > nh) a += sel_mass(x, m);
                });
                inbin_above += sel_block_sum(sm, a);
            }
        }
        // collect the candidates (counting them, with their key range)
        if (threadIdx.x == 0) {
            sm.n = 0u;
            sm.kmin = 0xFFFFFFFFu;
            sm.kmax = 0u;
        }
        __syncthreads();
        uint32_t lo = 0xFFFFFFFFu, hi = 0u;
        float am = 0.0f;
        each(hint, [&](float x, int) {
            const int bx = sel_bin1(x, m);
            if (bx > b1hi || !(x >= xmin)) return;
            if (bx < b1) {
                if (first) am += sel_mass(x, m);
                return;
            }
            const uint32_t kv = ord_key(x);
            if (kv >= klo && kv <= khi) {
                lo = min(lo, kv);
                hi = max(hi, kv);
                const uint32_t at = atomicAdd(&sm.n, 1u);
                if (at < static_cast<uint32_t>(kSelPool)) sm.pool_a()[at] = x;
            }
        });
        atomicMin(&sm.kmin, lo);
        atomicMax(&sm.kmax, hi);
        if (first) {
            above_mass = sel_block_sum(sm, am);  // (synchronises)
            if (mode == 1) ma = above_mass;      // the exact mass above the candidates
        }
        __syncthreads();
        first = false;
        n = sm.n;
        const uint32_t nlo = sm.kmin, nhi = sm.kmax;
        __syncthreads();
        if (n <= static_cast<uint32_t>(kSelPool)) break;
        klo = nlo;
        khi = nhi;
        big = true;
        if (klo == khi) {  // one value held by more tokens than fit
            gmass = static_cast<float>(n) * sel_mass(key_value(khi), m);
            return key_value(khi);
        }
    }
    // in shared memory: one finer level at a time down to a single value
    for (int pass = 0;; ++pass) {
        if (pass == kMaxPoolPasses) {
            gave_up = true;
            gmass = 0.0f;
            return -kInf;
        }
        if (threadIdx.x == 0) {
            sm.kmin = 0xFFFFFFFFu;
            sm.kmax = 0u;
        }
        __syncthreads();
        uint32_t lo = 0xFFFFFFFFu, hi = 0u;
        for (uint32_t e = threadIdx.x; e < n; e += kThreads) {
            const uint32_t kv = ord_key(sm.pool_a()[e]);
            lo = min(lo, kv);
            hi = max(hi, kv);
        }
        atomicMin(&sm.kmin, lo);
        atomicMax(&sm.kmax, hi);
        __syncthreads();
        klo = sm.kmin;
        khi = sm.kmax;
        __syncthreads();
        if (n == 0u || klo == khi) break;  // one value left
        const int sh = sel_shift(klo, khi);
        sel_clear(sm, kSelBins);
        __syncthreads();
        for (uint32_t e = threadIdx.x; e < n; e += kThreads) {
            const float x = sm.pool_a()[e];
            sel_add(sm, mode, sel_sub(ord_key(x), khi, sh), sel_mass(x, m));
        }
        __syncthreads();
        const int sb = sel_cross(sm, kSelBins, mode, k, target, ca, ma);
        uint32_t nlo = klo, nhi = khi;
        sel_narrow(nlo, nhi, sb, sh);
        if (threadIdx.x == 0) sm.n = 0u;
        __syncthreads();
        float a = 0.0f;
        for (uint32_t e = threadIdx.x; e < n; e += kThreads) {
            const float x = sm.pool_a()[e];
            const uint32_t kv = ord_key(x);
            if (kv >= nlo && kv <= nhi) sm.pool_b()[atomicAdd(&sm.n, 1u)] = x;
            else if (kv > nhi) a += sel_mass(x, m);
        }
        inbin_above += sel_block_sum(sm, a);  // (synchronises)
        n = sm.n;
        for (uint32_t e = threadIdx.x; e < n; e += kThreads) sm.pool_a()[e] = sm.pool_b()[e];
        __syncthreads();
    }
    const float xs = n ? key_value(khi) : -kInf;
    float gm = 0.0f;
    for (uint32_t e = threadIdx.x; e < n; e += kThreads) gm += sel_mass(sm.pool_a()[e], m);
    gmass = sel_block_sum(sm, gm);
    return xs;
}

// A lower bound of a row's threshold from its line maxima (lmx[0 .. nl), x units): mode 0
// (top-k): every token below the returned value has at least k line maxima, distinct tokens,
// above it; mode 1 (top-p): every token below it has line maxima of at least `target` mass above
// it (masses bounded from below by their 1/64-nat level-1 bin). The line maxima are counted into
// level-1 bins (copy 0 of the level-1 counts), the first bin whose cumulative count / mass bound
// reaches the goal is found, and the bound is the smallest line maximum in that bin or above.
// -inf when the line maxima alone never reach the goal (e.g. rows flat within their lines).
// Mode 2 (top-p, `target` = the mass (1 - P) Z that may lie below the kept set): y_e = m - e / 64
// for the smallest bin edge e whose upper bound of the mass of all tokens at or below y_e,
//   64 [ sum over lines in bins b >= e of e^(-b/64) + (lines in bins < e) e^(-e/64) ]
// (each line has at most 64 tokens, none above its maximum), stays within `target`: every token
// at or below y_e has at least Z - target = P Z of mass strictly above it, so it is dropped.
// sel_line_bound's mode 2, after the line maxima are counted into cnt[0 .. kSelBins1).
__device__ float sel_below_bound(SelSmem &sm, const uint32_t *cnt, float m, float budget, int per,
                                 int lane, int warp, int b0)
{
    __shared__ int s_edge;
    // this thread's bins: their counts and upper mass bounds (the last bin takes its lower edge)
    float tc = 0.0f, tm = 0.0f;
    for (int q = 0; q < per; ++q) {
        const float c = static_cast<float>(cnt[b0 + q]);
        tc += c;
        tm += c * sv::ex2_approx(-static_cast<float>(b0 + q) * (kLog2e / kSelBinsPerNat));
    }
    float ic = tc, im = tm;  // inclusive prefix sums over the threads, in bin order
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float yc = __shfl_up_sync(0xFFFFFFFFu, ic, o), ym = __shfl_up_sync(0xFFFFFFFFu, im, o);
        if (lane >= o) {
            ic += yc;
            im += ym;
        }
    }
    __shared__ float s_wc[kWarps], s_wm[kWarps];
    if (lane == 31) {
        s_wc[warp] = ic;
        s_wm[warp] = im;
    }
    if (threadIdx.x == 0) s_edge = INT_MAX;
    __syncthreads();
    float call = 0.0f, mall = 0.0f, cbef = ic - tc, mbef = im - tm;
    for (int w = 0; w < kWarps; ++w) {
        call += s_wc[w];
        mall += s_wm[w];
        if (w < warp) {
            cbef += s_wc[w];
            mbef += s_wm[w];
        }
    }
    // edge e = b0 + q: lines in bins < e counted in cb (before), the mass of bins >= e in ma
    float cb = cbef, mb = mbef;
    for (int q = 0; q < per; ++q) {
        const int e = b0 + q;
        const float ma = mall - mb;  // bins >= e
        const float ub = 64.0f * (ma + cb * sv::ex2_approx(-static_cast<float>(e) * (kLog2e / kSelBinsPerNat))) *
                         (1.0f + 0x1p-8f);  // margins for ex2 and the float sums
        if (ub <= budget) {
            atomicMin(&s_edge, e);
            break;
        }
        const float c = static_cast<float>(cnt[e]);
        cb += c;
        mb += c * sv::ex2_approx(-static_cast<float>(e) * (kLog2e / kSelBinsPerNat));
    }
    __syncthreads();
    const int e = s_edge;
    __syncthreads();
    // the edge value y_e = m - e / 64, rounded down (a smaller bound drops fewer tokens: safe)
    return e != INT_MAX ? __fsub_rd(m, static_cast<float>(e) * (1.0f / kSelBinsPerNat)) : -kInf;
}

__device__ float sel_line_bound(SelSmem &sm, const float *lmx, int nl, float m, int mode,
                                uint32_t k, float target)
{
    constexpr int per = kSelBins1 / kThreads;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, b0 = threadIdx.x * per;
    uint32_t *cnt = sm.cnt1();
    __shared__ int s_bin;
    __shared__ uint32_t s_kmin;
    for (int b = threadIdx.x; b < kSelBins1; b += kThreads) cnt[b] = 0u;
    if (threadIdx.x == 0) {
        s_bin = INT_MAX;
        s_kmin = 0xFFFFFFFFu;
    }
    __syncthreads();
    for (int q = threadIdx.x; q < nl; q += kThreads) {
        const float x = lmx[q];
        if (x == x) atomicAdd(cnt + sel_bin1(x, m), 1u);
    }
    __syncthreads();
    if (mode == 2) return sel_below_bound(sm, cnt, m, target, per, lane, warp, b0);
    auto value = [&](int b) {  // a bin's count, or a lower bound of its mass
        const float c = static_cast<float>(cnt[b]);
        if (mode == 0) return c;
        if (b == kSelBins1 - 1) return 0.0f;
        return c * sv::ex2_approx(-static_cast<float>(b + 1) * (kLog2e / kSelBinsPerNat)) *
               (1.0f - 0x1p-10f);
    };
    float t = 0.0f;
    for (int q = 0; q < per; ++q) t += value(b0 + q);
    float incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) sm.wm[warp] = incl;
    __syncthreads();
    float c = incl - t;  // before this thread's first bin
    for (int w = 0; w < warp; ++w) c += sm.wm[w];
    const float goal = mode == 0 ? static_cast<float>(k) : target;
    for (int q = 0; q < per; ++q) {
        c += value(b0 + q);
        if (c >= goal) {
            atomicMin(&s_bin, b0 + q);
            break;
        }
    }
    __syncthreads();
    const int bstar = s_bin;
    if (bstar != INT_MAX)
        for (int q = threadIdx.x; q < nl; q += kThreads) {
            const float x = lmx[q];
            if (x == x && sel_bin1(x, m) <= bstar) atomicMin(&s_kmin, ord_key(x));
        }
    __syncthreads();
    const float out = bstar != INT_MAX ? key_value(s_kmin) : -kInf;
    __syncthreads();
    return out;
}

// The threshold and the kept mass of every constrained row: one CTA per logit row. Rows without a
// penalty are read through their line maxima (sel_for_row_lines): a lower bound of the threshold
// from the line maxima alone (sel_line_bound), then passes that read only the lines and vectors
// that can reach the current bound. Penalised rows (whose line maxima are upper bounds, not
// values of tokens) read every element.
template <typename T, bool kPen>
__global__ void __launch_bounds__(kThreads, kPen ? 2 : 4)
sv_select_kernel(const T *__restrict__ logits, const T *__restrict__ lines,
                 const __grid_constant__ SelectParams P)
{
    __shared__ SelSmem sm;
    const int row = blockIdx.x, lane = threadIdx.x & 31;
    const int i = row_request(P.rq.cu, P.rq.n, row, lane);
    bool greedy;
    const float invT = request_invT(P.rq, i, greedy);
    int k;
    float Pp;
    if (!sel_active(P.top_k, P.top_p, i, P.V, greedy, k, Pp)) return;
    const bool use_k = k >= 1 && k < P.V, use_p = Pp < 1.0f;
    const int q0 = sv_ldg(P.rq.cu + i);
    const PenRow pr = kPen ? pen_row(P.pen, P.draft_ids, i, q0, row - q0 - i, P.V)
                           : PenRow{0.0f, nullptr, nullptr, 0};
    const T *rp = logits + static_cast<size_t>(row) * P.V;
    // the row maximum from the statistics partials (every warp the same)
    float L, s0;
    int idx;
    combine_row(P.part, row, P.V, P.maxseg, P.base_off, P.chunk, invT * kLog2e, L, s0, idx);
    const float m = __fmul_rn(L, invT);

    // the row's line maxima in x units, for rows without a penalty (every row of the kernel
    // without penalties: the host launches it with a line buffer of lmx_cap >= nl lines)
    const RowLines rl = row_lines(row, P.V, P.base_off);
    const bool by_lines = !kPen || (lines != nullptr && pr.f == 0.0f && rl.nl <= P.lmx_cap);
    float *lmx = sm.lmx();
    if (by_lines) {
        row_line_max<T, false>(rp, P.V, rl, lines, lmx, PenRow{0.0f, nullptr, nullptr, 0});
        __syncthreads();
        for (int q = threadIdx.x; q < rl.nl; q += kThreads) lmx[q] = __fmul_rn(lmx[q], invT);
        __syncthreads();
    }
    uint32_t *wq = sm.wq(P.lmx_cap);
    // the queued vectors' data in pool_b, which the row passes leave unused (kWarps * kSelQueue
    // 16-byte entries = kSelPool words)
    uint4 *wqd = reinterpret_cast<uint4 *>(sm.pool_b());
    auto each = [&](float xmin, auto &&f) {
        if constexpr (kPen) {
            if (!by_lines) {
                sel_for_row<T, kPen>(rp, P.V, invT, pr, f);
                return;
            }
        }
        sel_for_row_lines<T>(rp, P.V, invT, rl, lmx, xmin, wq, wqd, f);
    };

    // level 1: counts per bin of 1/64 nat (integer atomics) of the tokens x >= xmin
    auto count_level1 = [&](float xmin) {
        for (int b = threadIdx.x; b < kSel1Copies * kSelBins1; b += kThreads) sm.cnt1()[b] = 0u;
        __syncthreads();
        uint32_t *mine = sm.cnt1() + (threadIdx.x >> 7) * kSelBins1;  // four warps per copy
        bool done = false;
        if constexpr (kPen) {
            if (!by_lines) {
                sel_for_row<T, kPen>(rp, P.V, invT, pr, [&](float x, int) {
                    if (x >= xmin) atomicAdd(mine + sel_bin1(x, m), 1u);
                });
                done = true;
            }
        }
        if (!done) sel_count_lines<T>(rp, P.V, invT, m, rl, lmx, xmin, mine);
        __syncthreads();
    };
    float tau = -kInf, Z = s0, Sk = s0;  // Z: the mass of the top-k set, or of the row
    bool failed = false;
    // phase 0: top-k (its threshold, and Z = the mass of the kept set); phase 1: top-p within it.
    // One loop, so that the selection's code (sel_resolve with its row passes) exists once.
    for (int phase = use_k ? 0 : 1; phase <= (use_p ? 1 : 0); ++phase) {
        const float tk = tau;
        const float target = __fmul_rn(fmaxf(Pp, 1e-6f), Z);
        float xmin;
        if (phase == 0) {
            // the k-th largest token is at least the bound from the line maxima
            xmin = by_lines ? sel_line_bound(sm, lmx, rl.nl, m, 0, static_cast<uint32_t>(k), 0.0f) : -kInf;
        } else {
            // within a top-k set every kept token is at least tau_k; without one, bounds from the
            // line maxima (a lower bound of the mass above, an upper bound of the mass below)
            xmin = tk;
            if (!use_k && by_lines) {
                const float budget = __fmul_rd(__fmul_rd(__fsub_rd(1.0f, fmaxf(Pp, 1e-6f)), Z), 1.0f - 0x1p-10f);
                xmin = fmaxf(sel_line_bound(sm, lmx, rl.nl, m, 1, 0u, target),
                             sel_line_bound(sm, lmx, rl.nl, m, 2, 0u, budget));
            }
        }
        count_level1(xmin);
        uint32_t ca = 0u;
        float ma = 0.0f, above, inbin, gm;
        int blo, bhi;
        if (phase == 0) {
            blo = bhi = sel_cross(sm, kSelBins1, 0, static_cast<uint32_t>(k), 0.0f, ca, ma);
        } else {
            sel_bounds(sm, target, blo, bhi);
        }
        bool gave_up;
        const float t = sel_resolve(sm, each, m, blo, bhi, phase == 0 ? xmin : fmaxf(tk, xmin), phase,
                                    phase == 0 ? static_cast<uint32_t>(k) : 0u, phase == 0 ? 0.0f : target,
                                    ca, ma, above, inbin, gm, gave_up);
        tau = t;
        if (phase == 0) {
            Z = above + (inbin + gm);  // the bins above bk, then bk's tokens at or above tau_k
            Sk = Z;
        } else {
            Sk = ma + gm;
        }
        if (gave_up) failed = true;
    }
    if (failed) {  // (never expected) the row is left unconstrained and the call reports it
        tau = -kInf;
        Sk = s0;
        if (threadIdx.x == 0) atomicOr(P.flags + 1, SV_ERR_SELECT);
    }
    if (threadIdx.x == 0) {
        sv_st(P.sel_tau + row, tau);
        sv_st(P.sel_S + row, Sk);
    }
}

// ---------------------------------------------------------------------------------------
// 4. vocabulary shards: this rank holds columns [v0, v0 + Vs) of every row, v0 a multiple of 64
// ---------------------------------------------------------------------------------------
// Exchange 1: each row's statistics record, from the statistics partials of the shard.
template <typename T>
__global__ void __launch_bounds__(kThreads)
sv_shard_export_kernel(const T *__restrict__ logits, RequestTable rq,
                       const int32_t *__restrict__ draft_ids, const float *__restrict__ q,
                       const StatPart *__restrict__ part, int Vs, int v0, int maxseg,
                       int base_off, Divisor chunk, int R, spec_verify_shard_stat *__restrict__ out)
{
    const int lane = threadIdx.x & 31;
    const int row = static_cast<int>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (row >= R) return;  // whole warps
    const int i = row_request(rq.cu, rq.n, row, lane);
    const int q0 = sv_ldg(rq.cu + i), K = sv_ldg(rq.cu + i + 1) - q0, j = row - q0 - i;
    bool greedy;
    const float invT = request_invT(rq, i, greedy);
    float L, sx;
    int idx;
    combine_row(part, row, Vs, maxseg, base_off, chunk, invT * kLog2e, L, sx, idx);
    const int amax = resolve_argmax<T>(logits + static_cast<size_t>(row) * Vs, idx, L);
    if (lane == 0) {
        spec_verify_shard_stat rec;
        rec.max_logit = L;
        rec.sumexp = sx;
        rec.argmax = v0 + amax;
        rec.draft_logit = __int_as_float(0x7FC00000);
        rec.draft_prob = __int_as_float(0x7FC00000);
        rec.reserved = 0;
        if (j >= 0 && j < K && q0 + j < R - rq.n) {  // (a malformed cu_num_draft reads nothing)
            const int d = sv_ldg(draft_ids + q0 + j);
            if (d >= v0 && d < v0 + Vs) {
                rec.draft_logit = Elem<T>::at(logits + static_cast<size_t>(row) * Vs, d - v0);
                rec.draft_prob = q ? sv_ldg(q + static_cast<size_t>(q0 + j) * Vs + (d - v0)) : 1.0f;
            }
        }
        sv_st(out + row, rec);
    }
}

struct ShardParams {
    RequestTable rq;
    const int32_t *draft_ids;
    const float *q;                        // the shard's columns [nd, Vs], or nullptr
    const spec_verify_shard_stat *recs;    // [world][R]
    int world, R, V, Vs, v0, kmax, base_off;
    uint64_t seed;
    uint32_t req_base;
    spec_verify_shard_key *out;
};

// Exchange 2: combine every rank's records (rank order: the same numbers on every rank), take
// the acceptance decisions, and race this shard at the row of the first rejection. One CTA per
// request.
template <typename T>
__global__ void __launch_bounds__(kThreads, 2)
sv_shard_race_kernel(const T *__restrict__ logits, const T *__restrict__ lines,
                     const __grid_constant__ ShardParams P)
{
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ int s_js;
    __shared__ unsigned long long s_best;
    __shared__ int s_cnt;
    __shared__ int s_bin_n[kBins];
    __shared__ unsigned s_bin_max[kBins];
    __shared__ unsigned s_top;
    __shared__ uint32_t s_qgs[kWarps * kQueue];
    __shared__ float s_ql[kWarps * kQueue], s_qq[kWarps * kQueue];
    __shared__ unsigned long long s_wbk[kWarps];
    __shared__ int s_wbv[kWarps];
    const int i = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int q0 = sv_ldg(P.rq.cu + i), K = sv_ldg(P.rq.cu + i + 1) - q0;
    const VerifyLayout lay = verify_layout(P.Vs, P.kmax);
    {  // the batch must be consistent (as in the verify kernel); otherwise j* = -1: nothing emitted
        const int n = P.rq.n, nd = P.R - n;
        int bad = 0;
        for (int t = tid; t <= n; t += kThreads) {
            const int c0 = sv_ldg(P.rq.cu + t);
            if (t == 0) bad |= c0 != 0;
            if (t == n) bad |= c0 != nd;
            if (t < n) {
                const int c1 = sv_ldg(P.rq.cu + t + 1);
                bad |= (c1 < c0) | (static_cast<long long>(c1) - c0 > P.kmax) | (c0 < 0) | (c1 > nd);
            }
        }
        if (__syncthreads_or(bad)) {
            if (tid == 0) sv_st(P.out + i, spec_verify_shard_key{-1, -1, 0.0f, -1, 0.0f, -1});
            return;
        }
    }
    bool greedy;
    const float invT = request_invT(P.rq, i, greedy);
    const float c = invT * kLog2e;
    const uint32_t ireq = P.req_base + static_cast<uint32_t>(i);
    const int stride = P.kmax + 1;
    float *sm_m = reinterpret_cast<float *>(dyn + lay.rows), *sm_S = sm_m + stride;
    int *sm_amax = reinterpret_cast<int *>(sm_m + 2 * stride);
    if (tid == 0) s_js = K;
    __syncthreads();
    for (int j = warp; j <= K; j += kWarps) {
        const int row = q0 + i + j;
        float L = -kInf, sx = 0.0f, ld = __int_as_float(0x7FC00000), qd = ld;
        int idx = INT_MAX;
        for (int r = lane; r < P.world; r += 32) {
            const spec_verify_shard_stat rec = sv_ld(P.recs + static_cast<size_t>(r) * P.R + row);
            combine_stat(L, sx, idx, rec.max_logit, rec.sumexp, rec.argmax, c);
            if (rec.draft_logit == rec.draft_logit) {
                ld = rec.draft_logit;
                qd = rec.draft_prob;
            }
        }
        warp_reduce_stat(L, sx, idx, c);
        const unsigned own = __ballot_sync(0xFFFFFFFFu, ld == ld);
        if (own) {
            const int src = __ffs(own) - 1;
            ld = __shfl_sync(0xFFFFFFFFu, ld, src);
            qd = __shfl_sync(0xFFFFFFFFu, qd, src);
        }
        if (lane == 0) {
            const float m = __fmul_rn(L, invT);
            const int amax = idx == INT_MAX ? 0 : idx;
            sm_m[j] = m;
            sm_S[j] = sx;
            sm_amax[j] = amax;
            if (j < K) {
                const int d = sv_ldg(P.draft_ids + q0 + j);
                bool acc;
                if (greedy) {
                    acc = d == amax;  // [spec-notes] 8.3
                } else if (d < 0 || d >= P.V || !own) {
                    acc = false;
                } else {  // [spec-notes] answer code: q > 0 and p / q >= u
                    const float t_d = sv::exp_f32(__fsub_rn(__fmul_rn(ld, invT), m));
                    const sv::Philox4 u4 = sv::philox4x32_10(0u, static_cast<uint32_t>(j), ireq,
                                                             sv::kTagAccept,
                                                             static_cast<uint32_t>(P.seed),
                                                             static_cast<uint32_t>(P.seed >> 32));
                    acc = qd > 0.0f && __fdiv_rn(__fdiv_rn(t_d, sx), qd) >= sv::uniform_from_word(u4.x);
                }
                if (!acc) atomicMin(&s_js, j);
            }
        }
    }
    __syncthreads();
    const int js = s_js;
    spec_verify_shard_key o;
    o.jstar = js;
    o.token = greedy ? sm_amax[js] : -1;
    o.residual_key = 0.0f;
    o.residual_index = -1;
    o.p_key = 0.0f;
    o.p_index = -1;
    if (!greedy) {
        const int row = q0 + i + js;
        RaceRow<T> r;
        r.g0 = static_cast<uint32_t>(P.v0 / kGroup);
        r.rp = logits + static_cast<size_t>(row) * P.Vs;
        r.V = P.Vs;
        r.G = (P.Vs + kGroup - 1) / kGroup;
        r.m = sm_m[js];
        r.S = sm_S[js];
        r.invT = invT;
        r.j = static_cast<uint32_t>(js);
        r.ireq = ireq;
        r.k0 = static_cast<uint32_t>(P.seed);
        r.k1 = static_cast<uint32_t>(P.seed >> 32);
        r.dlrow = nullptr;
        r.md = 0.0f;
        r.Sd = 1.0f;
        r.pr = PenRow{0.0f, nullptr, nullptr, 0};
        r.tau = -kInf;
        r.qrow = nullptr;
        r.excl = -1;
        r.f64 = false;
        SearchSmem sm;
        sm.buf = reinterpret_cast<unsigned long long *>(dyn);
        sm.tmp = reinterpret_cast<unsigned long long *>(dyn + lay.tmp);
        sm.bin_n = s_bin_n;
        sm.bin_max = s_bin_max;
        sm.top = &s_top;
        sm.qgs = s_qgs;
        sm.ql = s_ql;
        sm.qq = s_qq;
        sm.lm = reinterpret_cast<float *>(dyn);
        sm.pb = reinterpret_cast<float *>(dyn + lay.pb);
        sm.ew = reinterpret_cast<uint32_t *>(dyn + lay.ew);
        sm.ag = dyn + lay.ag;
        sm.best = &s_best;
        sm.wbk = s_wbk;
        sm.wbv = s_wbv;
        sm.cnt = &s_cnt;
        const RowLines rl = row_lines(row, P.Vs, P.base_off);
        if (js < K) {  // the residual (with q) or the exclusion race (without) of this shard
            const bool residual = P.q != nullptr;
            const int d = sv_ldg(P.draft_ids + q0 + js);
            r.qrow = residual ? P.q + static_cast<size_t>(q0 + js) * P.Vs : nullptr;
            r.excl = (!residual && d >= P.v0 && d < P.v0 + P.Vs) ? d - P.v0 : -1;
            row_line_max<T, false>(r.rp, P.Vs, rl, lines, sm.lm, r.pr);
            __syncthreads();
            const unsigned long long b = residual ? race_search<T, true, false, false>(r, rl, sm)
                                                  : race_search<T, false, false, false>(r, rl, sm);
            if (b) {
                o.residual_key = key_dec(static_cast<unsigned>(b >> 32));
                o.residual_index = P.v0 + static_cast<int>(~static_cast<unsigned>(b));
            }
            r.qrow = nullptr;
            r.excl = -1;
            __syncthreads();
        }
        // the race over p: the bonus token, and the fallback of a residual empty on every
        // shard, which needs it only from shards whose own residual is empty
        if (js == K || o.residual_index < 0) {
            row_line_max<T, false>(r.rp, P.Vs, rl, lines, sm.lm, r.pr);
            __syncthreads();
            const unsigned long long b = race_search<T, false, false, false>(r, rl, sm);
            if (b) {
                o.p_key = key_dec(static_cast<unsigned>(b >> 32));
                o.p_index = P.v0 + static_cast<int>(~static_cast<unsigned>(b));
            }
        }
    }
    if (tid == 0) sv_st(P.out + i, o);
}

// The winner over the shards and the emitted row of each request (one thread per request).
__global__ void sv_shard_finish_kernel(const spec_verify_shard_key *__restrict__ races, int world,
                                       const int32_t *__restrict__ draft_ids,
                                       const int32_t *__restrict__ cu, int n, int kmax,
                                       int32_t *__restrict__ sampled,
                                       int32_t *__restrict__ num_sampled,
                                       int32_t *__restrict__ num_rejected)
{
    const int i = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
    if (i >= n) return;
    const int q0 = sv_ldg(cu + i), K = sv_ldg(cu + i + 1) - q0;
    const spec_verify_shard_key o0 = sv_ld(races + i);
    const int js = o0.jstar;
    const int stride = kmax + 1;
    if (js < 0 || js > K || K > kmax) {  // an inconsistent batch: nothing emitted
        for (int s = 0; s < stride; ++s) sv_st(sampled + static_cast<size_t>(i) * stride + s, -1);
        sv_st(num_sampled + i, 0);
        sv_st(num_rejected + i, 0);
        return;
    }
    int token = o0.token;
    if (token < 0) {
        unsigned long long best = 0ull;
        if (js < K)
            for (int r = 0; r < world; ++r) {
                const spec_verify_shard_key o = sv_ld(races + static_cast<size_t>(r) * n + i);
                if (o.residual_index >= 0) best = max(best, pack_key(o.residual_key, o.residual_index));
            }
        if (!best)
            for (int r = 0; r < world; ++r) {
                const spec_verify_shard_key o = sv_ld(races + static_cast<size_t>(r) * n + i);
                if (o.p_index >= 0) best = max(best, pack_key(o.p_key, o.p_index));
            }
        token = best ? static_cast<int>(~static_cast<unsigned>(best)) : 0;
    }
    int32_t *out = sampled + static_cast<size_t>(i) * stride;
    for (int s = 0; s < stride; ++s) sv_st(out + s, s < js ? sv_ldg(draft_ids + q0 + s) : (s == js ? token : -1));
    sv_st(num_sampled + i, js + 1);
    sv_st(num_rejected + i, K - js);
}

// One CTA per request. kDLMode: q comes from draft logits (P.dl); kPen: the batch has a
// frequency penalty. Separate instantiations, so that the plain path carries neither.
template <typename T, bool kDLMode, bool kPen>
__global__ void __launch_bounds__(kThreads, 2)
sv_verify_kernel(const T *__restrict__ logits, const T *__restrict__ lines,
                 const __grid_constant__ VerifyParams P)
{
    extern __shared__ __align__(16) unsigned char dyn[];
    __shared__ int s_js;
    __shared__ unsigned long long s_best;
    __shared__ int s_cnt;
    __shared__ int s_bin_n[kBins];
    __shared__ unsigned s_bin_max[kBins];
    __shared__ unsigned s_top;
    __shared__ uint32_t s_qgs[kWarps * kQueue];
    __shared__ float s_ql[kWarps * kQueue], s_qq[kWarps * kQueue];
    __shared__ unsigned long long s_wbk[kWarps];
    __shared__ int s_wbv[kWarps];
    const int i = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = P.rq.n;
    const int32_t *__restrict__ cu = P.rq.cu;
    const int stride = P.kmax + 1;
    const VerifyLayout lay = verify_layout(P.V, P.kmax);

    // 0. the batch must be consistent; every CTA checks all of cu_num_draft (small, in L2)
    const int q0 = sv_ldg(cu + i);
    const int K = sv_ldg(cu + i + 1) - q0;
    if (tid == 0) s_js = K;
    int bad = 0;
    for (int t = tid; t <= n; t += kThreads) {
        const int c0 = sv_ldg(cu + t);
        if (t == 0) bad |= c0 != 0;
        if (t == n) bad |= c0 != P.nd;
        if (t < n) {
            const int c1 = sv_ldg(cu + t + 1);
            bad |= (c1 < c0) | (static_cast<long long>(c1) - c0 > P.kmax) | (c0 < 0) | (c1 > P.nd);
        }
    }
    if (__syncthreads_or(bad)) {  // an inconsistent batch emits nothing for any request
        emit_row(i, -1, 0, 0, -1, nullptr, P.sampled, stride, P.num_sampled, P.num_rejected, tid,
                 kThreads);
        if (i == 0 && tid == 0) atomicOr(P.flags + 1, SV_ERR_BATCH);
        return;
    }
    const int row0 = q0 + i;
    bool greedy;
    const float invT = request_invT(P.rq, i, greedy);
    if (tid == 0 && pen_counts_row_bad(P.pen, i)) atomicOr(P.flags + 1, SV_ERR_COUNTS);
    const bool partial = P.partial && sv_ldg(P.partial + i) != 0;  // no token: only row stats
    const bool synthetic = P.nsyn > 0;
    const float c = invT * kLog2e;
    const uint32_t ireq = P.req_base + static_cast<uint32_t>(i);
    float *sm_m = reinterpret_cast<float *>(dyn + lay.rows), *sm_S = sm_m + stride;
    int *sm_amax = reinterpret_cast<int *>(sm_m + 2 * stride);
    float *sm_md = sm_m + 3 * stride, *sm_Sd = sm_m + 4 * stride;  // draft rows (draft logits)
    float *sm_tau = sm_m + 5 * stride;                              // sampling constraints
    int sel_k;
    float sel_p;
    const bool constrained = P.sel_tau && sel_active(P.rq.top_k, P.top_p, i, P.V, greedy, sel_k, sel_p);
    const T *dl = kDLMode ? static_cast<const T *>(P.dl) : nullptr;
    // this warp's first acceptance test: its inputs are read before the wait
    AcceptInputs ahead{false, 0, 0.0f, 1.0f};
    if (lane == 0 && warp < K && !partial && !synthetic && !greedy)
        ahead = accept_inputs<T>(logits + static_cast<size_t>(row0 + warp) * P.V, P.V, q0 + warp,
                                 P.draft_ids, P.q, dl);
    pdl_wait();  // the statistics partials and line maxima from here on

    // 1. row statistics from the partials (warp per row) and the acceptance tests
    for (int j = warp; j <= K; j += kWarps) {
        const int row = row0 + j;
        const long long rbase = static_cast<long long>(row) * P.V;
        float L, s;
        int idx;
        combine_row(P.part, row, P.V, P.maxseg, P.base_off, P.chunk, c, L, s, idx);
        float md = 0.0f, Sd = 1.0f;
        if (dl && j < K) {  // the draft row's q = softmax(draft logits / T): its m_d and S_d
            float Ld;
            int id;
            combine_row(P.dpart, q0 + j, P.V, P.maxseg, P.dbase_off, P.dchunk, c, Ld, Sd, id);
            md = __fmul_rn(Ld, invT);
        }
        float tau = -kInf;
        if (constrained) {  // the kept set and its mass, from the select kernel
            tau = sv_ldg(P.sel_tau + row);
            s = sv_ldg(P.sel_S + row);
        }
        // the argmax only where it is used: a greedy request's tests and output, the row output
        const int amax = greedy || P.opt_amax ? resolve_argmax<T>(logits + rbase, idx, L) : 0;
        if (lane == 0) {
            sm_md[j] = md;
            sm_Sd[j] = Sd;
            sm_tau[j] = tau;
            const float m = __fmul_rn(L, invT);  // = max_v fl(l_v / T): rounding is monotone
            sm_m[j] = m;
            sm_S[j] = s;
            sm_amax[j] = amax;
            if (P.opt_max) sv_st(P.opt_max + row, m);
            if (P.opt_sum) sv_st(P.opt_sum + row, s);
            if (P.opt_amax) sv_st(P.opt_amax + row, amax);
            if (j < K && !partial &&
                !(synthetic ? accept_synthetic(P, j, q0 + j, ireq)
                            : accept_draft<T>(logits + rbase, P.V, greedy, j, q0 + j,
                                              kPen ? pen_row(P.pen, P.draft_ids, i, q0, j, P.V)
                                                   : PenRow{0.0f, nullptr, nullptr, 0},
                                              invT, m, s, tau, amax, P.draft_ids, P.q, dl, md,
                                              Sd, P.seed, ireq,
                                              j == warp ? ahead : AcceptInputs{false, 0, 0.0f, 1.0f})))
                atomicMin(&s_js, j);
        }
    }
    __syncthreads();
    if (partial) {  // [MTP-eagle] get_num_sampled_and_rejected: chunked prefill emits nothing
        emit_row(i, -1, K, q0, -1, nullptr, P.sampled, stride, P.num_sampled, P.num_rejected, tid,
                 kThreads);
        return;
    }
    const int js = s_js;  // [MTP-eagle] _rejection_sample_kernel: first rejection, K if none
    if (greedy) {  // [spec-notes] 8.3: the target argmax at the mismatch, or of the bonus row
        emit_row(i, js, K, q0, sm_amax[js], P.draft_ids, P.sampled, stride, P.num_sampled,
                 P.num_rejected, tid, kThreads);
        return;
    }

    // 2. the race at j*
    const int row = row0 + js;
    RaceRow<T> r;
    r.g0 = 0u;
    r.rp = logits + static_cast<size_t>(row) * P.V;
    r.V = P.V;
    r.G = (P.V + kGroup - 1) / kGroup;
    r.m = sm_m[js];
    r.S = sm_S[js];
    r.invT = invT;
    r.j = static_cast<uint32_t>(js);
    r.ireq = ireq;
    r.k0 = static_cast<uint32_t>(P.seed);
    r.k1 = static_cast<uint32_t>(P.seed >> 32);
    r.f64 = P.f64 != 0;
    // synthetic mode: the token at j* is the target's own draw from p, nothing excluded
    const bool residual = !synthetic && js < K && (P.q != nullptr || dl != nullptr);
    r.qrow = residual && P.q ? P.q + static_cast<size_t>(q0 + js) * P.V : nullptr;
    r.dlrow = residual && dl ? dl + static_cast<size_t>(q0 + js) * P.V : nullptr;
    r.pr = kPen ? pen_row(P.pen, P.draft_ids, i, q0, js, P.V) : PenRow{0.0f, nullptr, nullptr, 0};
    r.tau = sm_tau[js];
    r.md = js < K ? sm_md[js] : 0.0f;
    r.Sd = js < K ? sm_Sd[js] : 1.0f;
    r.excl = (!synthetic && js < K && !residual) ? sv_ldg(P.draft_ids + q0 + js) : -1;
    SearchSmem sm;
    sm.buf = reinterpret_cast<unsigned long long *>(dyn);
    sm.tmp = reinterpret_cast<unsigned long long *>(dyn + lay.tmp);
    sm.bin_n = s_bin_n;
    sm.bin_max = s_bin_max;
    sm.top = &s_top;
    sm.qgs = s_qgs;
    sm.ql = s_ql;
    sm.qq = s_qq;
    sm.lm = reinterpret_cast<float *>(dyn);
    sm.pb = reinterpret_cast<float *>(dyn + lay.pb);
    sm.ew = reinterpret_cast<uint32_t *>(dyn + lay.ew);
    sm.ag = dyn + lay.ag;
    sm.best = &s_best;
    sm.wbk = s_wbk;
    sm.wbv = s_wbv;
    sm.cnt = &s_cnt;
    const RowLines rl = row_lines(row, P.V, P.base_off);
    row_line_max<T, kPen>(r.rp, P.V, rl, lines, sm.lm, r.pr);
    __syncthreads();
    unsigned long long best = residual ? race_search<T, true, kDLMode, kPen>(r, rl, sm)
                                       : race_search<T, false, false, kPen>(r, rl, sm);
    if (best == 0) {
        // nothing left of max(0, p - q) after rounding, or V == 1 with the only token rejected:
        // draw from p itself
        row_line_max<T, kPen>(r.rp, P.V, rl, lines, sm.lm, r.pr);
        __syncthreads();
        r.excl = -1;
        best = race_search<T, false, false, kPen>(r, rl, sm);
    }
    emit_row(i, js, K, q0, static_cast<int>(~static_cast<unsigned>(best)), P.draft_ids, P.sampled,
             stride, P.num_sampled, P.num_rejected, tid, kThreads);
}

// ---------------------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------------------
constexpr int kProfRing = 512;
constexpr int kKernels = 2;     // launches of a call without sampling constraints: stats, verify
constexpr int kProfSlots = 3;   // profiled kernels: stats, verify, select (top-k / top-p)
// static shared memory of a verify CTA besides the dynamic part (reserve)
constexpr int kVerifyStaticSmem = 10240;

struct ProfSlot {
    cudaEvent_t ev[kProfSlots + 1];  // before stats, after stats, after select, after verify
    bool pending;
};

int ceil_div(int a, int b) { return (a + b - 1) / b; }

// An NVTX range named after the entry point around each call, for profilers that attach an NVTX
// tool (Nsight Systems, Nsight Compute's --nvtx filters); without one it is a call into a no-op.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};

size_t verify_smem_bytes(int V, int kmax) { return verify_layout(V, kmax).total; }

}  // namespace

struct spec_verify_ctx {
    int device = 0;
    int max_num_reqs = 0, max_spec_len = 0, V = 0, dtype = SV_F32;
    int has_q = 0;       // draft probabilities may be given
    int has_dl = 0;      // draft logits may be given (spec_verify_run_draft_logits)
    int nsyn = 0;        // synthetic acceptance rates (0 = off)
    float syn[SV_MAX_SYNTHETIC] = {};
    int max_rows = 0, maxseg = 0;
    int stats_chunk = 0;   // 0: automatic (even split over whole waves)
    int stats_ctas = 1;      // one wave of the statistics kernel (SMs x CTAs per SM)
    int stats_ctas_pen = 1;  // one wave of its frequency-penalty instantiation
    StatPart *statpart = nullptr;
    StatPart *dpart = nullptr;  // partials of the draft rows (draft-logits mode)
    float *sel_tau = nullptr;   // [max_rows] top-k / top-p threshold per row
    float *sel_S = nullptr;     // [max_rows] kept mass per row
    void *lines = nullptr;      // largest logit of every 64-element line (logits dtype), or null
    uint32_t *penmask = nullptr;  // [max_num_reqs][ceil(V / 32) + 1] counts bits (frequency penalty)
    unsigned *flags = nullptr;  // [1] sticky error word
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
    double prof_ms[kProfSlots] = {0, 0, 0};
};

namespace {

long long stats_chunk_for(const spec_verify_ctx *ctx, long long all, bool pen)
{
    const long long wave = pen ? ctx->stats_ctas_pen : ctx->stats_ctas;
    auto aligned = [](long long c) {
        return std::max<long long>((c + kChunkAlign - 1) / kChunkAlign * kChunkAlign, kMinChunk);
    };
    long long chunk = ctx->stats_chunk;
    if (chunk <= 0) {
        // automatic: an even split over the fewest whole waves of CTAs whose chunk fits, one wave
        // when it can (measured faster than two on the bench workload: each CTA then runs one
        // long stream, and no second wave starts behind the first)
        for (long long waves = 1;; ++waves) {
            chunk = aligned((all + waves * wave - 1) / (waves * wave));
            if (chunk <= kMaxChunk) break;
        }
    }
    return std::min<long long>(aligned(chunk), kMaxChunk);
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
    cudaEventSynchronize(s.ev[kProfSlots]);
    // events: 0 before stats, 1 after it, 2 after select (right after 1 without it), 3 after verify
    float ms[kProfSlots] = {0.f, 0.f, 0.f};
    cudaEventElapsedTime(&ms[0], s.ev[0], s.ev[1]);
    cudaEventElapsedTime(&ms[2], s.ev[1], s.ev[2]);
    cudaEventElapsedTime(&ms[1], s.ev[2], s.ev[3]);
    for (int k = 0; k < kProfSlots; ++k) ctx->prof_ms[k] += ms[k];
    s.pending = false;
    ctx->prof_done++;
}

void free_all(spec_verify_ctx *ctx)
{
    cudaFree(ctx->statpart);
    cudaFree(ctx->dpart);
    cudaFree(ctx->sel_tau);
    cudaFree(ctx->sel_S);
    cudaFree(ctx->lines);
    cudaFree(ctx->penmask);
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

int optin_smem(int device)
{
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return v;
}

// Largest dynamic shared memory a verify CTA may use on `device`.
size_t verify_smem_limit(int device)
{
    return static_cast<size_t>(std::max(optin_smem(device) - kVerifyStaticSmem, 0));
}

// Allow the verify kernel the device's opt-in shared memory and report how many statistics
// CTAs fit on one SM (for the whole-wave grid).
template <typename T>
cudaError_t setup_kernels(int device, int *stats_per_sm, int *stats_pen_per_sm)
{
    const int limit = static_cast<int>(verify_smem_limit(device));
    // select: its fixed part and one row's line maxima; as much as a verify CTA may use
    cudaError_t es = cudaFuncSetAttribute(sv_select_kernel<T, false>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
    if (es == cudaSuccess)
        es = cudaFuncSetAttribute(sv_select_kernel<T, true>,
                                  cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
    if (es != cudaSuccess) return es;
    const void *kernels[] = {reinterpret_cast<const void *>(sv_shard_race_kernel<T>),
                             reinterpret_cast<const void *>(sv_verify_kernel<T, false, false>),
                             reinterpret_cast<const void *>(sv_verify_kernel<T, true, false>),
                             reinterpret_cast<const void *>(sv_verify_kernel<T, false, true>),
                             reinterpret_cast<const void *>(sv_verify_kernel<T, true, true>)};
    cudaError_t e = cudaSuccess;
    for (const void *k : kernels)
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, limit);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(stats_pen_per_sm, sv_stats_kernel<T, true>,
                                                      kThreads, 0);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(stats_per_sm, sv_stats_kernel<T, false>,
                                                         kThreads, 0);
}

// Statistics chunk for an array of `total` elements: the context's, or an even split over the
// fewest whole waves of CTAs that keeps a chunk within kMaxChunk (shared with any other array of
// the same launch).
long long stats_chunk_for(const spec_verify_ctx *ctx, long long all, bool pen);

template <typename T>
StatsArray<T> stats_array(const T *logits, long long total, long long chunk, int V, int draft_rows,
                          StatPart *part, T *lines)
{
    StatsArray<T> a;
    a.logits = logits;
    a.total = total;
    a.chunk = make_divisor(chunk);
    a.dv = make_divisor(V);
    a.base_off = static_cast<int>((reinterpret_cast<uintptr_t>(logits) % (kGroup * sizeof(T))) / sizeof(T));
    a.grid = total > 0 ? static_cast<int>((total + a.base_off + chunk - 1) / chunk) : 0;
    a.draft_rows = draft_rows;
    a.part = part;
    a.lines = lines;
    return a;
}

#ifdef SV_DEBUG_BOUNDS
// The arrays one call may touch, registered in g_dbg (stream-ordered) before its launches. The
// environment variable SV_DEBUG_SHRINK (bytes, default 0) leaves that many bytes of the end of
// the first registered array (the logits) out, so that tests can check that the check fires
// on memory the kernels may really read.
struct DbgList {
    DbgRanges r{};
    void add(const void *p, size_t bytes)
    {
        if (!p || bytes == 0 || r.n >= kDbgRanges) return;
        r.lo[r.n] = reinterpret_cast<unsigned long long>(p);
        r.hi[r.n] = r.lo[r.n] + bytes;
        r.n++;
    }
    int push(unsigned *flags, cudaStream_t stream)
    {
        r.flags = flags;
        if (const char *e = getenv("SV_DEBUG_SHRINK")) {
            const unsigned long long cut = strtoull(e, nullptr, 10);
            if (r.n > 0 && r.hi[0] - r.lo[0] > cut) r.hi[0] -= cut;
        }
        return cudaMemcpyToSymbolAsync(g_dbg, &r, sizeof(r), 0, cudaMemcpyHostToDevice, stream) ==
                       cudaSuccess ? SV_OK : SV_ECUDA;
    }
};

// The context's own scratch.
void dbg_add_ctx(DbgList &d, const spec_verify_ctx *ctx)
{
    const size_t rows = static_cast<size_t>(ctx->max_rows), seg = static_cast<size_t>(ctx->maxseg);
    const size_t eb = ctx->dtype == SV_BF16 ? 2 : 4, V = static_cast<size_t>(ctx->V);
    const size_t drows = static_cast<size_t>(ctx->max_num_reqs) * static_cast<size_t>(ctx->max_spec_len);
    d.add(ctx->statpart, rows * seg * kWarps * sizeof(StatPart));
    d.add(ctx->dpart, drows * seg * kWarps * sizeof(StatPart));
    d.add(ctx->sel_tau, rows * 4);
    d.add(ctx->sel_S, rows * 4);
    d.add(ctx->lines, (rows * V + 2 * kGroup) / kGroup * eb);
    if (ctx->penmask)
        d.add(ctx->penmask, static_cast<size_t>(ctx->max_num_reqs) * (static_cast<size_t>(ceil_div(ctx->V, 32)) + 1) * 4);
    d.add(ctx->flags, 2 * sizeof(unsigned));
}
#endif

// Both launches of one call (arguments already checked).
template <typename T>
int launch_all(spec_verify_ctx *ctx, const spec_verify_batch &b, const spec_verify_outputs &o,
               cudaStream_t stream)
{
    const T *logits = static_cast<const T *>(b.logits);
    const T *dl = b.num_draft_tokens > 0 ? static_cast<const T *>(b.draft_logits) : nullptr;
    const int num_reqs = b.num_reqs, nd = b.num_draft_tokens, kmax = b.max_spec_len_this_batch;
    const int32_t *cu = b.cu_num_draft;
    const int V = ctx->V;
    const int rows = nd + num_reqs;
    // statistics: the flattened [rows x V] logits (and [nd x V] draft logits) split evenly
    const long long total = static_cast<long long>(rows) * V;
    const long long total_d = dl ? static_cast<long long>(nd) * V : 0;
    const long long chunk1 = stats_chunk_for(ctx, total + total_d, b.frequency_penalty != nullptr);
    const RequestTable rq{cu, b.temperature, b.is_greedy, b.top_k, num_reqs};
    const int mask_stride = ceil_div(V, 32) + 1;
    const PenTable pen{b.frequency_penalty, b.output_bin_counts, b.counts_row, b.counts_rows, nd,
                       kmax, ctx->penmask, mask_stride};
    const bool pen_on = b.frequency_penalty != nullptr;
    T *lines = static_cast<T *>(ctx->lines);
    if (pen_on && !lines) return SV_EINVAL;  // the race's line maxima of a penalised row
    if (pen_on && !ctx->penmask) return SV_EINVAL;  // the statistics read the counts' bits
    const StatsArray<T> A = stats_array<T>(logits, total, chunk1, V, 0, ctx->statpart, lines);
    const StatsArray<T> D = stats_array<T>(dl, total_d, chunk1, V, 1, ctx->dpart, nullptr);
    const int base_off = A.base_off;

    VerifyParams P;
    P.rq = rq;
    P.draft_ids = b.draft_ids;
    P.q = b.draft_probs;
    P.dl = dl;
    P.dpart = ctx->dpart;
    P.dchunk = D.chunk;
    P.dbase_off = D.base_off;
    P.part = ctx->statpart;
    P.seed = b.seed;
    P.req_base = b.req_index_base;
    P.nd = nd;
    P.kmax = kmax;
    P.V = V;
    P.maxseg = ctx->maxseg;
    P.base_off = base_off;
    P.chunk = make_divisor(chunk1);
    P.sampled = o.sampled;
    P.num_sampled = o.num_sampled;
    P.num_rejected = o.num_rejected;
    P.opt_max = o.row_max;
    P.opt_sum = o.row_sumexp;
    P.opt_amax = o.row_argmax;
    P.flags = ctx->flags;
    P.partial = b.partial_prefill;
    P.pen = pen_on ? pen : PenTable{nullptr, nullptr, nullptr, 0};
    const bool sel_on = b.top_k != nullptr || b.top_p != nullptr;
    P.top_p = b.top_p;
    P.sel_tau = sel_on ? ctx->sel_tau : nullptr;
    P.sel_S = sel_on ? ctx->sel_S : nullptr;
    P.nsyn = ctx->nsyn;
    P.f64 = b.fp64_gumbel != 0;
    for (int k = 0; k < SV_MAX_SYNTHETIC; ++k) P.syn[k] = k < ctx->nsyn ? ctx->syn[k] : 0.0f;
    const size_t smem = verify_smem_bytes(V, kmax);

#ifdef SV_DEBUG_BOUNDS
    {
        const size_t n = static_cast<size_t>(num_reqs), R = static_cast<size_t>(rows);
        const size_t Vz = static_cast<size_t>(V), ndz = static_cast<size_t>(nd);
        DbgList d;
        d.add(logits, R * Vz * sizeof(T));
        d.add(b.draft_ids, ndz * 4);
        d.add(b.draft_probs, ndz * Vz * 4);
        d.add(b.draft_logits, ndz * Vz * sizeof(T));
        d.add(cu, (n + 1) * 4);
        d.add(b.temperature, n * 4);
        d.add(b.is_greedy, n);
        d.add(b.partial_prefill, n);
        d.add(b.frequency_penalty, n * 4);
        d.add(b.output_bin_counts, static_cast<size_t>(std::max(b.counts_rows, 0)) * Vz * 4);
        d.add(b.counts_row, n * 4);
        d.add(b.top_k, n * 4);
        d.add(b.top_p, n * 4);
        d.add(o.sampled, n * (static_cast<size_t>(kmax) + 1) * 4);
        d.add(o.num_sampled, n * 4);
        d.add(o.num_rejected, n * 4);
        d.add(o.row_max, R * 4);
        d.add(o.row_sumexp, R * 4);
        d.add(o.row_argmax, R * 4);
        dbg_add_ctx(d, ctx);
        if (d.push(ctx->flags, stream) != SV_OK) return SV_ECUDA;
    }
#endif
    ProfSlot *slot = nullptr;
    if (ctx->prof) {
        slot = &ctx->ring[static_cast<size_t>(ctx->prof_calls % kProfRing)];
        prof_collect(ctx, *slot);
        cudaEventRecord(slot->ev[0], stream);
    }
    const size_t smem1 = lines ? static_cast<size_t>(chunk1 / kGroup) * sizeof(T) : 0;
    if (pen_on && num_reqs > 0) {  // the counts' nonzero bits, read by the statistics
        const int bpr = ceil_div(mask_stride, kWarps * 32);
        sv_pen_mask_kernel<<<static_cast<unsigned>(num_reqs) * bpr, kThreads, 0, stream>>>(
            pen, num_reqs, V, bpr, ctx->penmask);
    }
    if (pen_on)
        sv_stats_kernel<T, true><<<A.grid + D.grid, kThreads, smem1, stream>>>(
            V, ctx->maxseg, A, D, rq, pen, b.draft_ids);
    else
        sv_stats_kernel<T, false><<<A.grid + D.grid, kThreads, smem1, stream>>>(
            V, ctx->maxseg, A, D, rq, PenTable{nullptr, nullptr, nullptr, 0}, b.draft_ids);
    if (slot) cudaEventRecord(slot->ev[1], stream);
    if (sel_on && !lines) return SV_EINVAL;  // the selection reads rows through their line maxima
    if (sel_on) {  // top-k / top-p: the kept set of every constrained row
        SelectParams SP;
        SP.rq = rq;
        SP.pen = P.pen;
        SP.draft_ids = b.draft_ids;
        SP.top_k = b.top_k;
        SP.top_p = b.top_p;
        SP.part = ctx->statpart;
        SP.V = V;
        SP.maxseg = ctx->maxseg;
        SP.base_off = base_off;
        SP.chunk = P.chunk;
        SP.sel_tau = ctx->sel_tau;
        SP.sel_S = ctx->sel_S;
        // the line maxima of one row (at most ceil(V / 64) + 1 lines) after the pools
        SP.lmx_cap = ceil_div(V, kGroup) + 2;
        SP.flags = ctx->flags;
        const size_t sel_smem = kSelDynSmem + static_cast<size_t>(SP.lmx_cap) * 4 +
                                static_cast<size_t>(kWarps) * kSelQueue * 4;
        if (pen_on)
            sv_select_kernel<T, true><<<rows, kThreads, sel_smem, stream>>>(logits, lines, SP);
        else
            sv_select_kernel<T, false><<<rows, kThreads, sel_smem, stream>>>(logits, lines, SP);
    }
    if (slot) cudaEventRecord(slot->ev[2], stream);
    auto verify = dl ? (pen_on ? sv_verify_kernel<T, true, true> : sv_verify_kernel<T, true, false>)
                     : (pen_on ? sv_verify_kernel<T, false, true> : sv_verify_kernel<T, false, false>);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_reqs));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaLaunchKernelEx(&cfg, verify, logits, lines, P);
    if (slot) {
        cudaEventRecord(slot->ev[3], stream);
        slot->pending = true;
        ctx->prof_calls++;
    }
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

// Device address of a host buffer that kernels can read in place: page-locked memory (allocated
// or registered through CUDA) is addressable from the device under unified addressing. nullptr
// for pageable memory, which is copied instead.
const void *in_place(const void *p)
{
    cudaPointerAttributes a;
    if (!p || cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        cudaGetLastError();
        return nullptr;
    }
    return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

// A batch with the arguments of the plain entry points; the other fields NULL / 0.
spec_verify_batch plain_batch(const void *logits, const int32_t *draft_ids, const float *q,
                              const void *dl, const int32_t *cu, const float *temperature,
                              const uint8_t *is_greedy, uint64_t seed, uint32_t base, int n,
                              int nd, int kmax)
{
    spec_verify_batch b{};
    b.logits = logits;
    b.draft_ids = draft_ids;
    b.draft_probs = q;
    b.draft_logits = dl;
    b.cu_num_draft = cu;
    b.temperature = temperature;
    b.is_greedy = is_greedy;
    b.seed = seed;
    b.req_index_base = base;
    b.num_reqs = n;
    b.num_draft_tokens = nd;
    b.max_spec_len_this_batch = kmax;
    return b;
}

// Host-visible argument checks of one call (nothing is launched when they fail); `aligned`:
// the arrays are the kernels' own (device) inputs, whose 16-byte alignment is required.
int check_run_args(const spec_verify_ctx *ctx, const spec_verify_batch &b,
                   const spec_verify_outputs &o, bool aligned = true)
{
    const int num_reqs = b.num_reqs, nd = b.num_draft_tokens, kmax = b.max_spec_len_this_batch;
    if (num_reqs < 0 || nd < 0 || kmax < 0) return SV_EINVAL;
    if (num_reqs > ctx->max_num_reqs || kmax > ctx->max_spec_len ||
        static_cast<long long>(nd) > static_cast<long long>(num_reqs) * kmax)
        return SV_ECAPACITY;
    if (num_reqs == 0) return SV_OK;
    if (!b.logits || !b.cu_num_draft || !b.temperature || !b.is_greedy || !o.sampled ||
        !o.num_sampled || !o.num_rejected || (nd > 0 && !b.draft_ids))
        return SV_EINVAL;
    if (b.draft_probs && !ctx->has_q) return SV_EINVAL;
    if (b.draft_logits && (!ctx->has_dl || b.draft_probs)) return SV_EINVAL;
    if ((b.frequency_penalty != nullptr) != (b.output_bin_counts != nullptr) ||
        (b.frequency_penalty && b.counts_rows < 1))
        return SV_EINVAL;
    if ((b.top_k || b.top_p) && !ctx->sel_tau) return SV_EINVAL;  // not in the static-scratch path
    if (aligned && (reinterpret_cast<uintptr_t>(b.logits) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(b.draft_probs) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(b.draft_logits) % 16 != 0))
        return SV_EINVAL;
    return SV_OK;
}

}  // namespace

extern "C" {

int spec_verify_init(spec_verify_ctx **out, int max_num_reqs, int max_spec_len, int vocab_size,
                     int logits_dtype, int draft_input, int device)
{
    if (!out) return SV_EINVAL;
    *out = nullptr;
    if (max_num_reqs <= 0 || max_spec_len < 0 || vocab_size <= 0) return SV_EINVAL;
    if (draft_input < 0 || draft_input > (SV_DRAFT_PROBS | SV_DRAFT_LOGITS)) return SV_EINVAL;
    if (logits_dtype != SV_F32 && logits_dtype != SV_BF16) return SV_EDTYPE;
    const long long rows = static_cast<long long>(max_num_reqs) * (max_spec_len + 1);
    const long long maxseg = ceil_div(vocab_size, kMinChunk) + 1;
    if (rows > INT_MAX / 8 || rows * maxseg * kWarps > (1LL << 31) || max_spec_len > (1 << 16) ||
        vocab_size >= (1 << 30))  // (argmax candidates hold 2 x an index in an int)
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
    // the raced row's group bounds must fit in one CTA's shared memory
    if (verify_smem_bytes(vocab_size, max_spec_len) > verify_smem_limit(device)) return SV_ECAPACITY;

    auto *ctx = new (std::nothrow) spec_verify_ctx();
    if (!ctx) return SV_ECAPACITY;
    ctx->device = device;
    ctx->max_num_reqs = max_num_reqs;
    ctx->max_spec_len = max_spec_len;
    ctx->V = vocab_size;
    ctx->dtype = logits_dtype;
    ctx->has_q = (draft_input & SV_DRAFT_PROBS) != 0;
    ctx->has_dl = (draft_input & SV_DRAFT_LOGITS) != 0;
    ctx->max_rows = static_cast<int>(rows);
    ctx->maxseg = static_cast<int>(maxseg);
    const size_t R = static_cast<size_t>(rows), S = static_cast<size_t>(maxseg);
    const size_t nlines = (R * static_cast<size_t>(vocab_size) + 2 * kGroup) / kGroup;
    const size_t eb = logits_dtype == SV_BF16 ? 2 : 4;
    bool ok = cudaMalloc(&ctx->statpart, R * S * kWarps * sizeof(StatPart)) == cudaSuccess &&
              cudaMalloc(&ctx->lines, nlines * eb) == cudaSuccess &&
              cudaMalloc(&ctx->flags, 2 * sizeof(unsigned)) == cudaSuccess;
    const size_t D = static_cast<size_t>(max_num_reqs) * static_cast<size_t>(max_spec_len);
    ok = ok && cudaMalloc(&ctx->sel_tau, R * sizeof(float)) == cudaSuccess &&
         cudaMalloc(&ctx->sel_S, R * sizeof(float)) == cudaSuccess;
    const size_t mask_words = static_cast<size_t>(max_num_reqs) * (static_cast<size_t>(ceil_div(vocab_size, 32)) + 1);
    ok = ok && cudaMalloc(&ctx->penmask, mask_words * sizeof(uint32_t)) == cudaSuccess;
    ok = ok && (!ctx->has_dl || D == 0 ||
                cudaMalloc(&ctx->dpart, D * S * kWarps * sizeof(StatPart)) == cudaSuccess);
    ok = ok && cudaMemset(ctx->flags, 0, 2 * sizeof(unsigned)) == cudaSuccess;
    int stats_per_sm = 0, stats_pen_per_sm = 0;
    ok = ok && (logits_dtype == SV_BF16 ? setup_kernels<uint16_t>(device, &stats_per_sm, &stats_pen_per_sm)
                                        : setup_kernels<float>(device, &stats_per_sm, &stats_pen_per_sm)) ==
                   cudaSuccess;
    ok = ok && cudaDeviceSynchronize() == cudaSuccess;
    if (!ok) {
        free_all(ctx);
        delete ctx;
        cudaGetLastError();
        return SV_ECUDA;
    }
    ctx->stats_ctas = std::max(stats_per_sm, 1) * prop.multiProcessorCount;
    ctx->stats_ctas_pen = std::max(stats_pen_per_sm, 1) * prop.multiProcessorCount;
    *out = ctx;
    return SV_OK;
}

int spec_verify_run_batch(spec_verify_ctx *ctx, const spec_verify_batch *batch,
                          const spec_verify_outputs *out, void *cuda_stream)
{
    const NvtxRange nvtx("spec_verify_run_batch");
    if (!ctx || !batch || !out) return SV_EINVAL;
    const int rc = check_run_args(ctx, *batch, *out);
    if (rc != SV_OK || batch->num_reqs == 0) return rc;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
    auto stream = static_cast<cudaStream_t>(cuda_stream);
    return ctx->dtype == SV_BF16 ? launch_all<uint16_t>(ctx, *batch, *out, stream)
                                 : launch_all<float>(ctx, *batch, *out, stream);
}

int spec_verify_run(spec_verify_ctx *ctx, const void *logits, const int32_t *draft_ids,
                    const float *draft_probs, const int32_t *cu_num_draft,
                    const float *temperature, const uint8_t *is_greedy, uint64_t seed,
                    uint32_t req_index_base, int num_reqs, int num_draft_tokens,
                    int max_spec_len_this_batch, int32_t *sampled, int32_t *num_sampled,
                    int32_t *num_rejected, float *opt_row_max, float *opt_row_sumexp,
                    int32_t *opt_row_argmax, void *cuda_stream)
{
    const spec_verify_batch b = plain_batch(logits, draft_ids, draft_probs, nullptr, cu_num_draft,
                                            temperature, is_greedy, seed, req_index_base,
                                            num_reqs, num_draft_tokens, max_spec_len_this_batch);
    const spec_verify_outputs o{sampled, num_sampled, num_rejected, opt_row_max, opt_row_sumexp,
                                opt_row_argmax};
    return spec_verify_run_batch(ctx, &b, &o, cuda_stream);
}

int spec_verify_run_draft_logits(spec_verify_ctx *ctx, const void *logits,
                                 const int32_t *draft_ids, const void *draft_logits,
                                 const int32_t *cu_num_draft, const float *temperature,
                                 const uint8_t *is_greedy, uint64_t seed,
                                 uint32_t req_index_base, int num_reqs, int num_draft_tokens,
                                 int max_spec_len_this_batch, int32_t *sampled,
                                 int32_t *num_sampled, int32_t *num_rejected, float *opt_row_max,
                                 float *opt_row_sumexp, int32_t *opt_row_argmax,
                                 void *cuda_stream)
{
    if (!ctx) return SV_EINVAL;
    if (!ctx->has_dl || (num_reqs > 0 && num_draft_tokens > 0 && !draft_logits)) return SV_EINVAL;
    const spec_verify_batch b = plain_batch(logits, draft_ids, nullptr, draft_logits, cu_num_draft,
                                            temperature, is_greedy, seed, req_index_base,
                                            num_reqs, num_draft_tokens, max_spec_len_this_batch);
    const spec_verify_outputs o{sampled, num_sampled, num_rejected, opt_row_max, opt_row_sumexp,
                                opt_row_argmax};
    return spec_verify_run_batch(ctx, &b, &o, cuda_stream);
}

int spec_verify_shard_stats(spec_verify_ctx *ctx, const void *logits_shard, int v0,
                            const int32_t *draft_ids, const float *draft_probs_shard,
                            const int32_t *cu_num_draft, const float *temperature,
                            const uint8_t *is_greedy, int num_reqs, int num_draft_tokens,
                            int max_spec_len_this_batch, spec_verify_shard_stat *out,
                            void *cuda_stream)
{
    const NvtxRange nvtx("spec_verify_shard_stats");
    if (!ctx || !out || v0 < 0 || v0 % kGroup != 0) return SV_EINVAL;
    const spec_verify_batch b = plain_batch(logits_shard, draft_ids, draft_probs_shard, nullptr,
                                            cu_num_draft, temperature, is_greedy, 0, 0, num_reqs,
                                            num_draft_tokens, max_spec_len_this_batch);
    int32_t dummy;
    const spec_verify_outputs o{&dummy, &dummy, &dummy, nullptr, nullptr, nullptr};
    int rc = check_run_args(ctx, b, o);
    if (rc != SV_OK || num_reqs == 0) return rc;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
    auto stream = static_cast<cudaStream_t>(cuda_stream);
    const int Vs = ctx->V, R = num_draft_tokens + num_reqs;
    const RequestTable rq{cu_num_draft, temperature, is_greedy, nullptr, num_reqs};
    const long long total = static_cast<long long>(R) * Vs;
    const long long chunk1 = stats_chunk_for(ctx, total, false);
#ifdef SV_DEBUG_BOUNDS
    {
        const size_t n = static_cast<size_t>(num_reqs), Rz = static_cast<size_t>(R);
        const size_t eb = ctx->dtype == SV_BF16 ? 2 : 4, ndz = static_cast<size_t>(num_draft_tokens);
        DbgList d;
        d.add(logits_shard, Rz * static_cast<size_t>(Vs) * eb);
        d.add(draft_ids, ndz * 4);
        d.add(draft_probs_shard, ndz * static_cast<size_t>(Vs) * 4);
        d.add(cu_num_draft, (n + 1) * 4);
        d.add(temperature, n * 4);
        d.add(is_greedy, n);
        d.add(out, Rz * sizeof(spec_verify_shard_stat));
        dbg_add_ctx(d, ctx);
        if (d.push(ctx->flags, stream) != SV_OK) return SV_ECUDA;
    }
#endif
    auto launch = [&](auto tag) -> int {
        using T = decltype(tag);
        const T *lg = static_cast<const T *>(logits_shard);
        T *lines = static_cast<T *>(ctx->lines);
        const StatsArray<T> A = stats_array<T>(lg, total, chunk1, Vs, 0, ctx->statpart, lines);
        const StatsArray<T> D = stats_array<T>(nullptr, 0, chunk1, Vs, 1, nullptr, nullptr);
        const size_t smem1 = static_cast<size_t>(chunk1 / kGroup) * sizeof(T);
        sv_stats_kernel<T, false><<<A.grid, kThreads, smem1, stream>>>(
            Vs, ctx->maxseg, A, D, rq, PenTable{nullptr, nullptr, nullptr, 0}, draft_ids);
        sv_shard_export_kernel<T><<<(R + kWarps - 1) / kWarps, kThreads, 0, stream>>>(
            lg, rq, draft_ids, draft_probs_shard, ctx->statpart, Vs, v0, ctx->maxseg, A.base_off,
            A.chunk, R, out);
        return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
    };
    return ctx->dtype == SV_BF16 ? launch(uint16_t{}) : launch(float{});
}

int spec_verify_shard_race(spec_verify_ctx *ctx, const void *logits_shard, int v0, int vocab_size,
                           const spec_verify_shard_stat *all_stats, int world,
                           const int32_t *draft_ids, const float *draft_probs_shard,
                           const int32_t *cu_num_draft, const float *temperature,
                           const uint8_t *is_greedy, uint64_t seed, uint32_t req_index_base,
                           int num_reqs, int num_draft_tokens, int max_spec_len_this_batch,
                           spec_verify_shard_key *out, void *cuda_stream)
{
    const NvtxRange nvtx("spec_verify_shard_race");
    if (!ctx || !out || !all_stats || world < 1 || v0 < 0 || v0 % kGroup != 0 ||
        vocab_size < v0 + ctx->V)
        return SV_EINVAL;
    const spec_verify_batch b = plain_batch(logits_shard, draft_ids, draft_probs_shard, nullptr,
                                            cu_num_draft, temperature, is_greedy, seed,
                                            req_index_base, num_reqs, num_draft_tokens,
                                            max_spec_len_this_batch);
    int32_t dummy;
    const spec_verify_outputs o{&dummy, &dummy, &dummy, nullptr, nullptr, nullptr};
    int rc = check_run_args(ctx, b, o);
    if (rc != SV_OK || num_reqs == 0) return rc;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
    auto stream = static_cast<cudaStream_t>(cuda_stream);
    ShardParams P;
    P.rq = RequestTable{cu_num_draft, temperature, is_greedy, nullptr, num_reqs};
    P.draft_ids = draft_ids;
    P.q = draft_probs_shard;
    P.recs = all_stats;
    P.world = world;
    P.R = num_draft_tokens + num_reqs;
    P.V = vocab_size;
    P.Vs = ctx->V;
    P.v0 = v0;
    P.kmax = max_spec_len_this_batch;
    P.seed = seed;
    P.req_base = req_index_base;
    P.out = out;
    const size_t smem = verify_smem_bytes(ctx->V, max_spec_len_this_batch);
#ifdef SV_DEBUG_BOUNDS
    {
        const size_t n = static_cast<size_t>(num_reqs), Rz = static_cast<size_t>(P.R);
        const size_t eb = ctx->dtype == SV_BF16 ? 2 : 4, ndz = static_cast<size_t>(num_draft_tokens);
        DbgList d;
        d.add(logits_shard, Rz * static_cast<size_t>(P.Vs) * eb);
        d.add(all_stats, static_cast<size_t>(world) * Rz * sizeof(spec_verify_shard_stat));
        d.add(draft_ids, ndz * 4);
        d.add(draft_probs_shard, ndz * static_cast<size_t>(P.Vs) * 4);
        d.add(cu_num_draft, (n + 1) * 4);
        d.add(temperature, n * 4);
        d.add(is_greedy, n);
        d.add(out, n * sizeof(spec_verify_shard_key));
        dbg_add_ctx(d, ctx);
        if (d.push(ctx->flags, stream) != SV_OK) return SV_ECUDA;
    }
#endif
    auto launch = [&](auto tag) -> int {
        using T = decltype(tag);
        const T *lg = static_cast<const T *>(logits_shard);
        P.base_off = static_cast<int>((reinterpret_cast<uintptr_t>(lg) % (kGroup * sizeof(T))) / sizeof(T));
        sv_shard_race_kernel<T><<<num_reqs, kThreads, smem, stream>>>(
            lg, static_cast<const T *>(ctx->lines), P);
        return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
    };
    return ctx->dtype == SV_BF16 ? launch(uint16_t{}) : launch(float{});
}

int spec_verify_shard_finish(spec_verify_ctx *ctx, const spec_verify_shard_key *all_races,
                             int world, const int32_t *draft_ids, const int32_t *cu_num_draft,
                             int num_reqs, int max_spec_len_this_batch, int32_t *sampled,
                             int32_t *num_sampled, int32_t *num_rejected, void *cuda_stream)
{
    const NvtxRange nvtx("spec_verify_shard_finish");
    if (!ctx || world < 1 || num_reqs < 0 || max_spec_len_this_batch < 0) return SV_EINVAL;
    if (num_reqs == 0) return SV_OK;
    if (!all_races || !cu_num_draft || !sampled || !num_sampled || !num_rejected) return SV_EINVAL;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
#ifdef SV_DEBUG_BOUNDS
    {
        const size_t n = static_cast<size_t>(num_reqs);
        DbgList d;
        d.add(all_races, static_cast<size_t>(world) * n * sizeof(spec_verify_shard_key));
        // draft ids: at most cu_num_draft[num_reqs] of them; the count is on the device, so the
        // whole capacity of the context is allowed
        d.add(draft_ids, static_cast<size_t>(ctx->max_num_reqs) * static_cast<size_t>(ctx->max_spec_len) * 4);
        d.add(cu_num_draft, (n + 1) * 4);
        d.add(sampled, n * (static_cast<size_t>(max_spec_len_this_batch) + 1) * 4);
        d.add(num_sampled, n * 4);
        d.add(num_rejected, n * 4);
        dbg_add_ctx(d, ctx);
        if (d.push(ctx->flags, static_cast<cudaStream_t>(cuda_stream)) != SV_OK) return SV_ECUDA;
    }
#endif
    sv_shard_finish_kernel<<<(num_reqs + kThreads - 1) / kThreads, kThreads, 0,
                             static_cast<cudaStream_t>(cuda_stream)>>>(
        all_races, world, draft_ids, cu_num_draft, num_reqs, max_spec_len_this_batch, sampled,
        num_sampled, num_rejected);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ECUDA;
}

int spec_verify_set_synthetic(spec_verify_ctx *ctx, const float *rates, int n)
{
    if (!ctx || n < 0 || n > SV_MAX_SYNTHETIC || (n > 0 && !rates)) return SV_EINVAL;
    for (int k = 0; k < n; ++k) {
        if (!(rates[k] >= 0.0f && rates[k] <= 1.0f)) return SV_EINVAL;
        if (k > 0 && rates[k] > rates[k - 1]) return SV_EINVAL;
    }
    for (int k = 0; k < SV_MAX_SYNTHETIC; ++k) ctx->syn[k] = k < n ? rates[k] : 0.0f;
    ctx->nsyn = n;
    return SV_OK;
}

int spec_verify_synthetic_rates(double mean_length, int num_spec, float *rates)
{
    if (num_spec < 0 || num_spec > SV_MAX_SYNTHETIC || (num_spec > 0 && !rates) ||
        !(mean_length >= 1.0 && mean_length <= num_spec + 1.0))
        return SV_EINVAL;
    const double accepted = mean_length - 1.0;  // mean number of accepted drafts
    const double whole = std::floor(accepted);
    for (int j = 0; j < num_spec; ++j)
        rates[j] = j < whole ? 1.0f : (j == static_cast<int>(whole) ? static_cast<float>(accepted - whole) : 0.0f);
    return SV_OK;
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
    const NvtxRange nvtx("spec_verify_run_host");
    if (!ctx) return SV_EINVAL;
    if (!ctx->io_logits) return SV_EINVAL;
    // the device path's checks, less alignment: host arrays are staged or read in place
    const spec_verify_batch hb = plain_batch(logits, draft_ids, draft_probs, nullptr, cu_num_draft,
                                             temperature, is_greedy, seed, req_index_base,
                                             num_reqs, num_draft_tokens, max_spec_len_this_batch);
    const spec_verify_outputs ho{sampled, num_sampled, num_rejected, nullptr, nullptr, nullptr};
    int rc = check_run_args(ctx, hb, ho, false);
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
    // the verifier reads only a few entries of q: page-locked q is read in place, not copied
    const float *q_dev = static_cast<const float *>(in_place(draft_probs));
    bool ok = cudaMemcpyAsync(ctx->io_logits, logits, rows * V * eb, cudaMemcpyHostToDevice, stream) == cudaSuccess &&
              (!draft_probs || q_dev ||
               cudaMemcpyAsync(ctx->io_q, draft_probs, static_cast<size_t>(num_draft_tokens) * V * 4,
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
    rc = spec_verify_run(ctx, ctx->io_logits, d_ids, draft_probs ? (q_dev ? q_dev : ctx->io_q) : nullptr, d_cu,
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

int spec_verify_get_profile(spec_verify_ctx *ctx, double *ms, int64_t *calls)
{
    if (!ctx || !ms || !calls) return SV_EINVAL;
    DeviceGuard g(ctx->device);
    if (!g.ok) return SV_EDEVICE;
    for (auto &s : ctx->ring) prof_collect(ctx, s);
    for (int k = 0; k < kProfSlots; ++k) {
        ms[k] = ctx->prof_ms[k];
        ctx->prof_ms[k] = 0.0;
    }
    *calls = ctx->prof_done;
    ctx->prof_done = 0;
    return SV_OK;
}

int spec_verify_set_chunks(spec_verify_ctx *ctx, int stats_chunk)
{
    if (!ctx || stats_chunk < -1) return SV_EINVAL;
    if (stats_chunk == -1) ctx->stats_chunk = 0;
    else if (stats_chunk) ctx->stats_chunk = (std::max(stats_chunk, kMinChunk) + kChunkAlign - 1) / kChunkAlign * kChunkAlign;
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
// with the fixed chunk a row spans at most this many statistics CTAs
constexpr int kNoAllocMaxSeg = (kNoAllocMaxVocab + kFixedChunk - 1) / kFixedChunk + 1;

constexpr size_t align256(size_t x) { return (x + 255) / 256 * 256; }
constexpr size_t kOffStatPart = 0;
constexpr size_t kOffFlags =
    kOffStatPart + align256(sizeof(StatPart) * size_t(kNoAllocMaxRows) * kNoAllocMaxSeg * kWarps);
constexpr size_t kNoAllocBytes = kOffFlags + align256(2 * sizeof(unsigned));

// One copy per device that loads this library, kept until the process exits. Every call of
// spec_verify_run_noalloc on a device shares it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
struct NoAllocDevice {
    void *base = nullptr;     // device address of g_noalloc_scratch on this device
    size_t smem_limit = 0;    // largest dynamic shared memory of a verify CTA here
};
NoAllocDevice g_noalloc_dev[kNoAllocMaxDevices];

// Set-up of device `dev` (current), once per device and then cached: the device must be an
// sm_103 part; the device address of the static scratch is looked up (the host-side name of
// the array is not a device address); the kernels' shared-memory limits are set. Later calls
// only read the cache, so a call on a device already set up makes no CUDA runtime query.
int noalloc_device(int dev, NoAllocDevice *out)
{
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoAllocDevice &d = g_noalloc_dev[dev];
    if (!d.base) {
        int major = 0, minor = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
            cudaGetLastError();
            return SV_EDEVICE;
        }
        if (major != 10 || minor != 3) return SV_EDEVICE;  // built for sm_103a only
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return SV_ECUDA;
        }
        int a = 0;
        int b = 0;
        if (setup_kernels<uint16_t>(dev, &a, &b) != cudaSuccess || setup_kernels<float>(dev, &a, &b) != cudaSuccess) {
            cudaGetLastError();
            return SV_ECUDA;
        }
        d.smem_limit = verify_smem_limit(dev);
        d.base = p;
    }
    *out = d;
    return SV_OK;
}

// The current device, if it is one this entry point can keep state for.
int noalloc_current(int *dev)
{
    if (cudaGetDevice(dev) != cudaSuccess || *dev < 0 || *dev >= kNoAllocMaxDevices) {
        cudaGetLastError();
        return SV_EDEVICE;
    }
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
    const NvtxRange nvtx("spec_verify_run_noalloc");
    if (logits_dtype != SV_F32 && logits_dtype != SV_BF16) return SV_EDTYPE;
    if (vocab_size <= 0 || num_reqs < 0 || num_draft_tokens < 0 || max_spec_len_this_batch < 0)
        return SV_EINVAL;
    if (vocab_size > kNoAllocMaxVocab || num_reqs > kNoAllocMaxReqs ||
        static_cast<long long>(num_draft_tokens) + num_reqs > kNoAllocMaxRows ||
        max_spec_len_this_batch >= kNoAllocMaxRows ||
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
    int rc = noalloc_current(&dev);
    if (rc != SV_OK) return rc;
    NoAllocDevice nd;
    rc = noalloc_device(dev, &nd);
    if (rc != SV_OK) return rc;
    if (verify_smem_bytes(vocab_size, max_spec_len_this_batch) > nd.smem_limit) return SV_ECAPACITY;
    auto *bytes = static_cast<unsigned char *>(nd.base);

    // A context on the host stack whose scratch pointers are carved from the static array; the
    // fixed statistics chunk keeps every row within kNoAllocMaxSeg partials. There is no room for
    // line maxima: the verify kernel takes them from the raced rows themselves.
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
    view.statpart = reinterpret_cast<StatPart *>(bytes + kOffStatPart);
    view.flags = reinterpret_cast<unsigned *>(bytes + kOffFlags);
    auto stream = static_cast<cudaStream_t>(cuda_stream);
    const spec_verify_batch b = plain_batch(logits, draft_ids, draft_probs, nullptr, cu_num_draft,
                                            temperature, is_greedy, seed, req_index_base,
                                            num_reqs, num_draft_tokens, max_spec_len_this_batch);
    const spec_verify_outputs o{sampled, num_sampled, num_rejected, opt_row_max, opt_row_sumexp,
                                opt_row_argmax};
    return logits_dtype == SV_BF16 ? launch_all<uint16_t>(&view, b, o, stream)
                                   : launch_all<float>(&view, b, o, stream);
}

extern "C" int spec_verify_noalloc_last_error(uint32_t *err_word)
{
    if (!err_word) return SV_EINVAL;
    int dev = -1;
    int rc = noalloc_current(&dev);
    if (rc != SV_OK) return rc;
    NoAllocDevice nd;
    rc = noalloc_device(dev, &nd);
    if (rc != SV_OK) return rc;
    unsigned *word = reinterpret_cast<unsigned *>(static_cast<unsigned char *>(nd.base) + kOffFlags) + 1;
    unsigned w = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&w, word, sizeof(unsigned), cudaMemcpyDeviceToHost) != cudaSuccess ||
        cudaMemset(word, 0, sizeof(unsigned)) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
        return SV_ECUDA;
    *err_word = w;
    return SV_OK;
}
