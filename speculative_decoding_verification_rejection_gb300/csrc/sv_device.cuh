// Device-side random numbers and binary32 elementary functions of the verification sampler.
//
// Race clocks: tokens come in groups of 64 (group g = v >> 6, slot s = v & 63). Philox counter
// (g, j, request, kClockHead) gives W (word 0) and the slot a (word 1 & 63) that holds the
// group's smallest clock E_g = -log(W) / 64; slot s != a has clock E_g - log(U_s), U_s word
// s & 3 of counter (g, j, request, kClockHead + 1 + s / 4). By the memoryless property of the
// exponential the 64 clocks are i.i.d. Exp(1), and E_g bounds every key of the group.
//
// Every decision of the sampler (acceptance test, race keys) is defined with these functions,
// so they use only correctly rounded binary32 operations written as explicit intrinsics
// (__fmaf_rn, __fmul_rn, __fadd_rn, __fsub_rn, __fdiv_rn): the compiler may not contract or
// reorder them, and the result is fixed bit for bit by the algorithm below.
#pragma once

#include <cstdint>

namespace sv {

// ---------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3",
// SC'11): ten rounds; a round multiplies counter words 0 and 2 by the two round multipliers,
// mixes the high halves with the other counter words and the key, and the key is advanced by
// the two Weyl increments (golden ratio and sqrt(3) - 1 in 32-bit fixed point).
// ---------------------------------------------------------------------------------------
struct Philox4 {
    uint32_t x, y, z, w;
};

__device__ __forceinline__ Philox4 philox4x32_10(uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                                                 uint32_t k0, uint32_t k1)
{
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t lo0 = 0xD2511F53u * c0;
        const uint32_t hi0 = __umulhi(0xD2511F53u, c0);
        const uint32_t lo1 = 0xCD9E8D57u * c2;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
        c0 = hi1 ^ c1 ^ k0;
        c1 = lo1;
        c2 = hi0 ^ c3 ^ k1;
        c3 = lo0;
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return Philox4{c0, c1, c2, c3};
}

// U in (0,1) from a 32-bit word: (floor(w / 2^9) + 1/2) * 2^-23, exact in binary32.
__device__ __forceinline__ float uniform_from_word(uint32_t w)
{
    return __fmul_rn(__fadd_rn(__uint2float_rn(w >> 9), 0.5f), 0x1p-23f);
}

// Counter word 3 of the acceptance uniform, of a race group's head call, and of its sixteen
// slot calls (kClockHead + 1 + slot / 4).
constexpr uint32_t kTagAccept = 0u;
constexpr uint32_t kClockHead = 8u;

// ---------------------------------------------------------------------------------------
// binary32 exp: Cody & Waite (1980) reduction d = k ln2 + r with k = round(d log2 e) taken by
// adding 1.5 * 2^23 in one fused multiply-add, r reduced with a two-part ln 2, exp(r) by its
// degree-7 Taylor polynomial in Horner form, result exp(r) * 2^k. Defined as 0 below -87.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float exp_f32(float d)
{
    if (!(d >= -87.0f)) return d != d ? d : 0.0f;
    if (d > 88.0f) return __int_as_float(0x7F800000);
    const float shifter = 0x1.8p+23f;
    const float kf = __fsub_rn(__fmaf_rn(d, 0x1.715476p+0f, shifter), shifter);
    float r = __fmaf_rn(-kf, 0x1.62e430p-1f, d);     // ln 2 rounded to binary32
    r = __fmaf_rn(-kf, -0x1.05c610p-29f, r);          // the remainder of ln 2
    float p = 0x1.a01a02p-13f;                         // 1/7!
    p = __fmaf_rn(p, r, 0x1.6c16c2p-10f);              // 1/6!
    p = __fmaf_rn(p, r, 0x1.111112p-7f);               // 1/5!
    p = __fmaf_rn(p, r, 0x1.555556p-5f);               // 1/4!
    p = __fmaf_rn(p, r, 0x1.555556p-3f);               // 1/3!
    p = __fmaf_rn(p, r, 0.5f);
    p = __fmaf_rn(p, r, 1.0f);
    p = __fmaf_rn(p, r, 1.0f);
    const int k = __float2int_rn(kf);
    return __fmul_rn(p, __int_as_float((k + 127) << 23));
}

// ---------------------------------------------------------------------------------------
// binary32 log for x > 0: x = 2^k f with f in [sqrt(1/2), sqrt(2)), ln f = 2 atanh(s),
// s = (f - 1) / (f + 1), summed as 2s + s z (2/3 + z (2/5 + z (2/7 + z 2/9))), z = s^2;
// ln x = k ln 2 + ln f with a two-part ln 2. Subnormals are scaled by 2^23 first.
// 0 -> -inf, negative or NaN -> NaN, +inf -> +inf.
// ---------------------------------------------------------------------------------------
__device__ __forceinline__ float log_f32(float x)
{
    if (x != x || x < 0.0f) return __int_as_float(0x7FC00000);
    if (x == 0.0f) return __int_as_float(0xFF800000);
    if (x == __int_as_float(0x7F800000)) return x;
    int k = 0;
    uint32_t b = __float_as_uint(x);
    if (b < 0x00800000u) {
        b = __float_as_uint(__fmul_rn(x, 0x1p+23f));
        k = -23;
    }
    k += static_cast<int>(b >> 23) - 127;
    uint32_t fb = (b & 0x007FFFFFu) | 0x3F800000u;
    if (fb > 0x3FB504F3u) {  // f > sqrt(2): halve it
        fb -= 0x00800000u;
        k += 1;
    }
    const float f = __uint_as_float(fb);
    const float g = __fsub_rn(f, 1.0f);
    const float s = __fdiv_rn(g, __fadd_rn(g, 2.0f));
    const float z = __fmul_rn(s, s);
    float P = __fmaf_rn(z, 0x1.c71c72p-3f, 0x1.24924ap-2f);  // 2/9, 2/7
    P = __fmaf_rn(z, P, 0x1.99999ap-2f);                      // 2/5
    P = __fmaf_rn(z, P, 0x1.555556p-1f);                      // 2/3
    const float R = __fmul_rn(z, P);
    const float lnf = __fmaf_rn(s, R, __fadd_rn(s, s));
    const float kf = __int2float_rn(k);
    return __fmaf_rn(kf, 0x1.62e430p-1f, __fmaf_rn(kf, -0x1.05c610p-29f, lnf));
}

// ---------------------------------------------------------------------------------------
// Race clocks in binary64 (the fp64 Gumbel option): the same group layout with 52-bit uniforms.
// Counter (g, j, request, kClockHead64) gives W = uniform64(word 0, word 1) and the slot
// a = word 2 & 63 of the group's smallest clock E_g = -log(W) / 64; slot s != a has clock
// E_g + (-log U_s), U_s = uniform64 of words (0, 1) (even s) or (2, 3) (odd s) of counter
// (g, j, request, kClockHead64 + 1 + s / 2).
// ---------------------------------------------------------------------------------------
constexpr uint32_t kClockHead64 = 32u;

// U in (0,1) from two words: (m + 1/2) * 2^-52, m = hi * 2^20 + (lo >> 12); exact in binary64.
__device__ __forceinline__ double uniform64_from_words(uint32_t hi, uint32_t lo)
{
    const unsigned long long m = (static_cast<unsigned long long>(hi) << 20) | (lo >> 12);
    return __dmul_rn(__dadd_rn(__ull2double_rn(m), 0.5), 0x1p-52);
}

// binary64 log for x > 0, the binary32 log's method in double: x = 2^k f with f in
// [sqrt(1/2), sqrt(2)), ln f = 2 atanh(s), s = (f - 1) / (f + 1), summed as 2s + s z P(z),
// z = s^2, P(z) = 2/3 + z (2/5 + ... + z 2/19) (the series 2 s^(2n+1) / (2n+1) to n = 9; the
// first term left out is below 0.15 ulp of the result); ln x = k ln 2 + ln f with ln 2 split
// into a 42-bit part (k ln2_hi exact) and its binary64 remainder. Subnormals are scaled by 2^54
// first. 0 -> -inf, negative or NaN -> NaN, +inf -> +inf.
__device__ __forceinline__ double log_f64(double x)
{
    if (x != x || x < 0.0) return __longlong_as_double(0x7FF8000000000000ll);
    if (x == 0.0) return __longlong_as_double(static_cast<long long>(0xFFF0000000000000ull));
    if (x == __longlong_as_double(0x7FF0000000000000ll)) return x;
    int k = 0;
    unsigned long long b = static_cast<unsigned long long>(__double_as_longlong(x));
    if (b < 0x0010000000000000ull) {
        b = static_cast<unsigned long long>(__double_as_longlong(__dmul_rn(x, 0x1p+54)));
        k = -54;
    }
    k += static_cast<int>(b >> 52) - 1023;
    unsigned long long fb = (b & 0x000FFFFFFFFFFFFFull) | 0x3FF0000000000000ull;
    if (fb > 0x3FF6A09E667F3BCCull) {  // f > sqrt(2): halve it
        fb -= 0x0010000000000000ull;
        k += 1;
    }
    const double f = __longlong_as_double(static_cast<long long>(fb));
    const double g = __dsub_rn(f, 1.0);
    const double s = __ddiv_rn(g, __dadd_rn(g, 2.0));
    const double z = __dmul_rn(s, s);
    double P = __fma_rn(z, 0x1.af286bca1af28p-4, 0x1.e1e1e1e1e1e1ep-4);  // 2/19, 2/17
    P = __fma_rn(z, P, 0x1.1111111111111p-3);                             // 2/15
    P = __fma_rn(z, P, 0x1.3b13b13b13b14p-3);                             // 2/13
    P = __fma_rn(z, P, 0x1.745d1745d1746p-3);                             // 2/11
    P = __fma_rn(z, P, 0x1.c71c71c71c71cp-3);                             // 2/9
    P = __fma_rn(z, P, 0x1.2492492492492p-2);                             // 2/7
    P = __fma_rn(z, P, 0x1.999999999999ap-2);                             // 2/5
    P = __fma_rn(z, P, 0x1.5555555555555p-1);                             // 2/3
    const double R = __dmul_rn(z, P);
    const double lnf = __fma_rn(s, R, __dadd_rn(s, s));
    const double kf = static_cast<double>(k);
    return __fma_rn(kf, 0x1.62e42fefa3800p-1, __fma_rn(kf, 0x1.ef35793c76730p-45, lnf));
}

// Fast 2^x (MUFU), for sums and for conservative screening only -- never for a decision.
__device__ __forceinline__ float ex2_approx(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

}  // namespace sv
