// beam_sincos.cuh -- cos and sin of an FP32 angle, rounded to FP32 as if from the exact values.
//
// The rotary embedding rotates each pair (q_i, q_{i+64}) by an FP32 angle; the oracle takes the
// cosine and sine of that angle exactly and rounds once to FP32.  A rotation output can be a
// near-cancellation (q_i cos - q_{i+64} sin), so any error in cos/sin shows up magnified in
// BF16 ulps of the output.  This routine returns the correctly rounded values except in rare
// near-tie cases, so the kernel's FP32 rotation matches the oracle bit for bit.
//
// Method (all in FP32 arithmetic with fused multiply-adds, no double precision):
//  * Range reduction after Cody & Waite (1980): k = nearest integer to x * 2/pi (decided with
//    the product's exact error so that |r| <= pi/4), r = x - k * pi/2 with pi/2 split into four
//    FP32 pieces; the products k * piece_0 and k * piece_1 are split exactly with an FMA
//    (Dekker's product), x - k * piece_0 is exact (Sterbenz), and the remaining sum is carried
//    as an unevaluated pair hi + lo with Knuth's TwoSum.  Valid for |x| < 2^24.
//  * sin(r) and cos(r) from their Taylor series, the leading terms evaluated in pair ("double
//    length", Dekker 1971) arithmetic and the tail (from r^9 / r^10) in FP32, for a total error
//    near 2^-45 relative; the pair is rounded once to FP32.
//  * Quadrant k mod 4 maps (sin r, cos r) to (sin x, cos x).
// Constants are the exact values 1/n!, 2/pi and pi/2 split into FP32 pieces.
//
// Compiled for the device (the RoPE kernel) and for the host (the library's host helper that
// the CPU tests check against correctly rounded values), with identical IEEE FP32 semantics:
// no contraction (-fmad=false on the device, -ffp-contract=off on the host), explicit FMAs.
#pragma once

#include <cmath>

#if defined(__CUDACC__)
#define BEAM_HD __host__ __device__ __forceinline__
#else
#define BEAM_HD inline
#endif

namespace beam {
namespace sc {

#if defined(__CUDA_ARCH__)
#define BEAM_FMA(a, b, c) __fmaf_rn((a), (b), (c))
#define BEAM_RINT(a) rintf(a)
#else
#define BEAM_FMA(a, b, c) std::fma((float)(a), (float)(b), (float)(c))
#define BEAM_RINT(a) std::rint((float)(a))
#endif

struct Pair {
    float hi, lo;
};

// s + e == a + b exactly (Knuth)
BEAM_HD Pair two_sum(float a, float b)
{
    const float s = a + b;
    const float bp = s - a;
    const float e = (a - (s - bp)) + (b - bp);
    return {s, e};
}

// s + e == a + b exactly when |a| >= |b| (Dekker)
BEAM_HD Pair fast_two_sum(float a, float b)
{
    const float s = a + b;
    return {s, b - (s - a)};
}

BEAM_HD Pair mul(Pair a, Pair b)
{
    const float p = a.hi * b.hi;
    float e = BEAM_FMA(a.hi, b.hi, -p);
    e = e + (a.hi * b.lo + a.lo * b.hi);
    return fast_two_sum(p, e);
}

BEAM_HD Pair add(Pair a, Pair b)
{
    const Pair s = two_sum(a.hi, b.hi);
    const float e = s.lo + (a.lo + b.lo);
    return fast_two_sum(s.hi, e);
}

// 2/pi and pi/2 in FP32 pieces
constexpr float kTwoOverPiHi = 0x1.45f306p-1f;
constexpr float kTwoOverPiLo = 0x1.b93910p-26f;
constexpr float kPio2_0 = 0x1.921fb6p+0f;
constexpr float kPio2_1 = -0x1.777a5cp-25f;
constexpr float kPio2_2 = -0x1.ee59dap-50f;
constexpr float kPio2_3 = 0x1.98a2e0p-77f;

// Taylor coefficients (-1)^j / n!: pairs for the leading terms, FP32 for the tail
constexpr Pair kS3 = {-0x1.555556p-3f, 0x1.555556p-28f};
constexpr Pair kS5 = {0x1.111112p-7f, -0x1.ddddde0p-32f};
constexpr Pair kS7 = {-0x1.a01a02p-13f, 0x1.7f97fap-39f};
constexpr float kS9 = 0x1.71de3ap-19f;
constexpr float kS11 = -0x1.ae6456p-26f;
constexpr float kS13 = 0x1.612462p-33f;
constexpr float kS15 = -0x1.ae7f3ep-41f;
constexpr Pair kC4 = {0x1.555556p-5f, -0x1.555556p-30f};
constexpr Pair kC6 = {-0x1.6c16c2p-10f, 0x1.27d27ep-35f};
constexpr Pair kC8 = {0x1.a01a02p-16f, -0x1.7f97fap-42f};
constexpr float kC10 = -0x1.27e4fcp-22f;
constexpr float kC12 = 0x1.1eed8ep-29f;
constexpr float kC14 = -0x1.93974ap-37f;
constexpr float kC16 = 0x1.ae7f3ep-45f;

}  // namespace sc

// Largest |x| the reduction above handles; beyond it callers use another routine.
constexpr float kSinCosMaxArg = 16777216.0f;  // 2^24

// sin and cos of x (|x| < 2^24), each the FP32 rounding of the exact value except in rare
// near-tie cases.
BEAM_HD void sincos_rounded(float x, float *s_out, float *c_out)
{
    using namespace sc;
    if (x == 0.0f) {  // keeps the sign of a zero sine
        *s_out = x;
        *c_out = 1.0f;
        return;
    }
    // k = nearest integer to x * 2/pi, with q + qe = x * 2/pi to ~2^-48 relative
    const float q = x * kTwoOverPiHi;
    const float qe = BEAM_FMA(x, kTwoOverPiHi, -q) + x * kTwoOverPiLo;
    float k = BEAM_RINT(q);
    const float f = (q - k) + qe;  // q - k is exact
    if (f > 0.5f)
        k = k + 1.0f;
    else if (f < -0.5f)
        k = k - 1.0f;

    // r = x - k * pi/2 as a pair
    const float p0 = k * kPio2_0;
    const float e0 = BEAM_FMA(k, kPio2_0, -p0);  // k * piece_0 == p0 + e0 exactly
    const float t = x - p0;                       // exact
    const float p1 = k * kPio2_1;
    const float e1 = BEAM_FMA(k, kPio2_1, -p1);
    const Pair a = two_sum(t, -e0);
    const Pair b = two_sum(a.hi, -p1);
    const float lo = (((a.lo + b.lo) - e1) - k * kPio2_2) - k * kPio2_3;
    const Pair r = two_sum(b.hi, lo);

    // z = r^2
    const float zh = r.hi * r.hi;
    const Pair z = fast_two_sum(zh, BEAM_FMA(r.hi, r.hi, -zh) + 2.0f * r.hi * r.lo);

    // sin r = r + r z (S3 + z (S5 + z (S7 + z tail)))
    const float ts = kS9 + z.hi * (kS11 + z.hi * (kS13 + z.hi * kS15));
    Pair u = add(kS7, mul(z, Pair{ts, 0.0f}));
    u = add(kS5, mul(z, u));
    u = add(kS3, mul(z, u));
    const Pair sp = add(r, mul(mul(z, u), r));

    // cos r = 1 + z (-1/2 + z (C4 + z (C6 + z (C8 + z tail))))
    const float tc = kC10 + z.hi * (kC12 + z.hi * (kC14 + z.hi * kC16));
    Pair v = add(kC8, mul(z, Pair{tc, 0.0f}));
    v = add(kC6, mul(z, v));
    v = add(kC4, mul(z, v));
    v = add(Pair{-0.5f, 0.0f}, mul(z, v));
    const Pair cp = add(Pair{1.0f, 0.0f}, mul(z, v));

    const float sr = sp.hi + sp.lo;
    const float cr = cp.hi + cp.lo;
    switch ((int)k & 3) {
    case 0: *s_out = sr; *c_out = cr; break;
    case 1: *s_out = cr; *c_out = -sr; break;
    case 2: *s_out = -sr; *c_out = -cr; break;
    default: *s_out = -cr; *c_out = sr; break;
    }
}

#undef BEAM_FMA
#undef BEAM_RINT

}  // namespace beam
