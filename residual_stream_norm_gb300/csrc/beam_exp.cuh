// beam_exp.cuh -- correctly rounded FP32 exp and the FP32 sigmoid built on it (host and device).
//
// The routing kernel ranks experts by sigmoid scores, so the sigmoid must be reproducible bit
// for bit: sigma(z) = 1 / (1 + RN32(exp(-z))), an FP32 add and an IEEE division, with
// RN32(exp) the FP32 rounding of the exact exponential.
//
// exp(x) = 2^k exp(r), k = rint(x log2 e), r = x - k ln 2.  ln 2 is split into three FP32
// pieces: the first has 15 significant bits, so k * L0 is exact for |k| <= 2^8 and x - k * L0
// is exact too (its bits all lie on x's or k * L0's grid, within 24 of each other).  r is then
// carried as an FP32 pair (hi, lo), and exp(r) is the Taylor series to degree 12, in FP32 pair
// ("double-float") arithmetic:
//   - TwoSum and Dekker's FMA TwoProduct are exact;
//   - each pair operation is accurate to a few 2^-46;
//   - the series remainder for |r| <= 0.36 is below 2^-51.
// The pair is rounded once to FP32.  When the pair lies within kExpBand (2^-40 relative, a
// generous bound on its error) of a rounding boundary, the value is recomputed in FP64
// double-double (series to degree 22, error near 2^-100) and rounded from there.  That happens
// for about 2^-16 of arguments.
//
// Constants: L0, L1, L2 are ln 2 split into FP32 pieces (each the FP32 rounding of what
// remains); the series coefficients are 1/n! as FP32 pairs (hi = RN32(1/n!), lo =
// RN32(1/n! - hi)), and as FP64 pairs for the fallback.
#pragma once

#include <cmath>
#include <cstdint>
#include <cstring>

#if defined(__CUDACC__)
#define BEAM_XP_HD __host__ __device__ __forceinline__
#else
#define BEAM_XP_HD inline
#endif

namespace beam {
namespace xp {

// --- IEEE operations with explicit rounding (never contracted) ---------------------------------

BEAM_XP_HD float fadd(float a, float b)
{
#if defined(__CUDA_ARCH__)
    return __fadd_rn(a, b);
#else
    return a + b;
#endif
}
BEAM_XP_HD float fsub(float a, float b)
{
#if defined(__CUDA_ARCH__)
    return __fsub_rn(a, b);
#else
    return a - b;
#endif
}
BEAM_XP_HD float fmul(float a, float b)
{
#if defined(__CUDA_ARCH__)
    return __fmul_rn(a, b);
#else
    return a * b;
#endif
}
BEAM_XP_HD float ffma(float a, float b, float c)
{
#if defined(__CUDA_ARCH__)
    return __fmaf_rn(a, b, c);
#else
    return std::fmaf(a, b, c);
#endif
}
BEAM_XP_HD float fdiv(float a, float b)
{
#if defined(__CUDA_ARCH__)
    return __fdiv_rn(a, b);
#else
    return a / b;
#endif
}
BEAM_XP_HD double dadd(double a, double b)
{
#if defined(__CUDA_ARCH__)
    return __dadd_rn(a, b);
#else
    return a + b;
#endif
}
BEAM_XP_HD double dsub(double a, double b)
{
#if defined(__CUDA_ARCH__)
    return __dsub_rn(a, b);
#else
    return a - b;
#endif
}
BEAM_XP_HD double dmul(double a, double b)
{
#if defined(__CUDA_ARCH__)
    return __dmul_rn(a, b);
#else
    return a * b;
#endif
}
BEAM_XP_HD double dfma(double a, double b, double c)
{
#if defined(__CUDA_ARCH__)
    return __fma_rn(a, b, c);
#else
    return std::fma(a, b, c);
#endif
}
BEAM_XP_HD float bits_f(uint32_t u)
{
#if defined(__CUDA_ARCH__)
    return __uint_as_float(u);
#else
    float f;
    std::memcpy(&f, &u, sizeof f);
    return f;
#endif
}
BEAM_XP_HD double bits_d(uint64_t u)
{
#if defined(__CUDA_ARCH__)
    return __longlong_as_double((long long)u);
#else
    double d;
    std::memcpy(&d, &u, sizeof d);
    return d;
#endif
}
BEAM_XP_HD uint32_t f_bits(float f)
{
#if defined(__CUDA_ARCH__)
    return __float_as_uint(f);
#else
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return u;
#endif
}

// --- FP32 pair ("double-float") arithmetic ------------------------------------------------------

struct F2 {
    float hi, lo;
};

BEAM_XP_HD F2 two_sum(float a, float b)
{
    const float s = fadd(a, b);
    const float bp = fsub(s, a);
    return F2{s, fadd(fsub(a, fsub(s, bp)), fsub(b, bp))};
}
BEAM_XP_HD F2 fast_two_sum(float a, float b)  // |a| >= |b|
{
    const float s = fadd(a, b);
    return F2{s, fsub(b, fsub(s, a))};
}
BEAM_XP_HD F2 f2_add(F2 a, F2 b)
{
    const F2 s = two_sum(a.hi, b.hi);
    return fast_two_sum(s.hi, fadd(s.lo, fadd(a.lo, b.lo)));
}
BEAM_XP_HD F2 f2_mul(F2 a, F2 b)
{
    const float p = fmul(a.hi, b.hi);
    const float e = ffma(a.hi, b.hi, -p);  // exact error of the product
    return fast_two_sum(p, fadd(e, fadd(fmul(a.hi, b.lo), fmul(a.lo, b.hi))));
}

// 1/n! as FP32 pairs, n = 0..12
BEAM_XP_HD F2 inv_fact_f2(int n)
{
    switch (n) {
    case 0: case 1: return F2{1.0f, 0.0f};
    case 2: return F2{0.5f, 0.0f};
    case 3: return F2{bits_f(0x3e2aaaabu), bits_f(0xb1aaaaabu)};
    case 4: return F2{bits_f(0x3d2aaaabu), bits_f(0xb0aaaaabu)};
    case 5: return F2{bits_f(0x3c088889u), bits_f(0xafeeeeefu)};
    case 6: return F2{bits_f(0x3ab60b61u), bits_f(0xae13e93fu)};
    case 7: return F2{bits_f(0x39500d01u), bits_f(0xac3fcbfdu)};
    case 8: return F2{bits_f(0x37d00d01u), bits_f(0xaabfcbfdu)};
    case 9: return F2{bits_f(0x3638ef1du), bits_f(0x292ad8e6u)};
    case 10: return F2{bits_f(0x3493f27eu), bits_f(0xa808760au)};
    case 11: return F2{bits_f(0x32d7322bu), bits_f(0x25fea89cu)};
    default: return F2{bits_f(0x310f76c7u), bits_f(0x24ff8d89u)};
    }
}

// --- FP64 pair ("double-double") fallback --------------------------------------------------------

struct D2 {
    double hi, lo;
};

BEAM_XP_HD D2 d_two_sum(double a, double b)
{
    const double s = dadd(a, b);
    const double bp = dsub(s, a);
    return D2{s, dadd(dsub(a, dsub(s, bp)), dsub(b, bp))};
}
BEAM_XP_HD D2 d_fast_two_sum(double a, double b)
{
    const double s = dadd(a, b);
    return D2{s, dsub(b, dsub(s, a))};
}
BEAM_XP_HD D2 d2_add(D2 a, D2 b)
{
    const D2 s = d_two_sum(a.hi, b.hi);
    const D2 t = d_two_sum(a.lo, b.lo);
    const D2 u = d_fast_two_sum(s.hi, dadd(s.lo, t.hi));
    return d_fast_two_sum(u.hi, dadd(u.lo, t.lo));
}
BEAM_XP_HD D2 d2_mul(D2 a, D2 b)
{
    const double p = dmul(a.hi, b.hi);
    const double e = dfma(a.hi, b.hi, -p);
    return d_fast_two_sum(p, dadd(e, dadd(dmul(a.hi, b.lo), dmul(a.lo, b.hi))));
}

// 1/n! as FP64 pairs, n = 0..22
BEAM_XP_HD D2 inv_fact_d2(int n)
{
    constexpr uint64_t kHi[23] = {
        0x3ff0000000000000ull, 0x3ff0000000000000ull, 0x3fe0000000000000ull,
        0x3fc5555555555555ull, 0x3fa5555555555555ull, 0x3f81111111111111ull,
        0x3f56c16c16c16c17ull, 0x3f2a01a01a01a01aull, 0x3efa01a01a01a01aull,
        0x3ec71de3a556c734ull, 0x3e927e4fb7789f5cull, 0x3e5ae64567f544e4ull,
        0x3e21eed8eff8d898ull, 0x3de6124613a86d09ull, 0x3da93974a8c07c9dull,
        0x3d6ae7f3e733b81full, 0x3d2ae7f3e733b81full, 0x3ce952c77030ad4aull,
        0x3ca6827863b97d97ull, 0x3c62f49b46814157ull, 0x3c1e542ba4020225ull,
        0x3bd71b8ef6dcf572ull, 0x3b90ce396db7f853ull};
    constexpr uint64_t kLo[23] = {
        0x0ull, 0x0ull, 0x0ull,
        0x3c65555555555555ull, 0x3c45555555555555ull, 0x3c01111111111111ull,
        0xbbef49f49f49f49full, 0x3b6a01a01a01a01aull, 0x3b3a01a01a01a01aull,
        0xbb6c154f8ddc6c00ull, 0x3b3cbbc05b4fa99aull, 0xbafc062e06d1f209ull,
        0xbac2aec959e14c06ull, 0x3a8f28e0cc748ebeull, 0x3a305d6f8a2efd1full,
        0x39e1d8656b0ee8cbull, 0x39a1d8656b0ee8cbull, 0x398ac981465ddc6cull,
        0x394eec01221a8b0bull, 0x38f2650f61dbdcb4ull, 0x387ea72b4afe3c2full,
        0xb87d043ae40c4647ull, 0xb83aebcdbd20331cull};
    return D2{bits_d(kHi[n]), bits_d(kLo[n])};
}

// exp(x) for |x| <= 89 as an FP64 pair (error near 2^-100 relative), times 2^-k.
BEAM_XP_HD D2 exp_reduced_d2(float x, int k)
{
    const D2 ln2 = {bits_d(0x3fe62e42fefa39efull), bits_d(0x3c7abc9e3b39803full)};
    const D2 kl = d2_mul(D2{(double)k, 0.0}, ln2);
    const D2 r = d2_add(D2{(double)x, 0.0}, D2{-kl.hi, -kl.lo});
    D2 p = inv_fact_d2(22);
    for (int n = 21; n >= 0; --n)
        p = d2_add(d2_mul(p, r), inv_fact_d2(n));
    return p;
}

// FP32 rounding (nearest even) of hi + lo for an FP64 pair with |lo| <= ulp(hi) / 2.
BEAM_XP_HD float d2_to_f32(D2 a)
{
    float f = (float)a.hi;  // nearest
    const double back = (double)f;
    const double diff = dadd(dsub(a.hi, back), a.lo);  // a - f, exact enough
    // neighbours of f and the midpoints towards them
    const float up = bits_f(f_bits(f) + 1u), dn = bits_f(f_bits(f) - 1u);
    const double half_up = dmul(dsub((double)up, back), 0.5);
    const double half_dn = dmul(dsub(back, (double)dn), 0.5);
    if (diff > half_up || (diff == half_up && (f_bits(f) & 1u)))
        f = up;
    else if (-diff > half_dn || (-diff == half_dn && (f_bits(f) & 1u)))
        f = dn;
    return f;
}

}  // namespace xp

constexpr float kExpBand = 9.094947017729282e-13f;  // 2^-40

// RN32(exp(x)) for FP32 x in [-17, 90]: exact rounding (below -17 the caller needs no value).
// Results past the FP32 range are +inf.
BEAM_XP_HD float exp_rounded(float x)
{
    using namespace xp;
    if (x > 89.0f)
        return bits_f(0x7f800000u);
    const float L0 = bits_f(0x3f317200u), L1 = bits_f(0x35bfbe8eu), L2 = bits_f(0x29779abdu);
    const float log2e = bits_f(0x3fb8aa3bu);
    const float kf = rintf(fmul(x, log2e));
    const int k = (int)kf;
    // r = x - k ln2 as an FP32 pair: x - k L0 is exact; k L1 by an exact TwoProduct
    const float a = fsub(x, fmul(kf, L0));
    const float p1 = fmul(kf, L1);
    const float p1e = ffma(kf, L1, -p1);
    F2 r = two_sum(a, -p1);
    r = fast_two_sum(r.hi, fsub(fsub(r.lo, p1e), fmul(kf, L2)));
    // exp(r) by Horner's rule on the Taylor series in FP32 pairs
    F2 p = inv_fact_f2(12);
#pragma unroll
    for (int n = 11; n >= 0; --n)
        p = f2_add(f2_mul(p, r), inv_fact_f2(n));
    // round once; recompute in FP64 pairs when within the band of a rounding boundary
    float f = fadd(p.hi, p.lo);
    const uint32_t u = f_bits(f);
    const float ulp_half_up = bits_f(((u >> 23) - 24u) << 23);
    const float ulp_half_dn = (u & 0x7fffffu) ? ulp_half_up : bits_f(((u >> 23) - 25u) << 23);
    const float band = fmul(f, kExpBand);
    const float res = fadd(fsub(p.hi, f), p.lo);  // p - f
    if (res > fsub(ulp_half_up, band) || res < fsub(band, ulp_half_dn))
        f = d2_to_f32(exp_reduced_d2(x, k));
    // f * 2^k in two exact steps (k <= 129; the second step may overflow to +inf)
    const int k1 = k / 2, k2 = k - k1;
    return fmul(fmul(f, bits_f((uint32_t)(127 + k1) << 23)), bits_f((uint32_t)(127 + k2) << 23));
}

// The FP32 sigmoid 1 / (1 + RN32(exp(-z))).  Below -z = -17, exp(-z) < 2^-24 and 1 + it rounds to
// 1 whatever its value, so no exponential is formed there.
BEAM_XP_HD float sigmoid_rounded(float z)
{
    using namespace xp;
    if (z != z)
        return z;
    const float x = -z;
    const float e = x < -17.0f ? 0.0f : exp_rounded(x);
    return fdiv(1.0f, fadd(1.0f, e));
}

}  // namespace beam
