// beam_f32x2.cuh -- packed FP32 pair arithmetic (sm_100+ add/mul/fma .f32x2) for the
// boundary-path kernels, and the residual operand rule shared with the host.
//
// Each .f32x2 instruction applies the IEEE round-to-nearest FP32 operation to both lanes, so a
// packed computation gives bit-for-bit the results of the scalar one at half the instruction
// count.  A pair holds BF16 elements 2i (low lane) and 2i+1 (high lane) of one 32-bit word.
//
// Caution: the compiler fuses a packed product that feeds a packed add/sub into one packed FMA
// (the product is then not rounded), despite the .rn modifiers and even through an opaque move.
// Packed products therefore only feed packed adds where the product is exact (squares of BF16
// values).  An inexact product followed by an add is formed either with the scalar __fmul_rn /
// __fadd_rn intrinsics, which are never fused, or as a packed fma(x, y, nz) whose addend nz is
// -0 held in a launch parameter: the rounded product exactly (a zero product keeps its sign),
// and an FMA followed by an add is not fused.
#pragma once

#include <cmath>
#include <cstdint>
#include <cstring>

namespace beam {

// ---------------------------------------------------------------------------------------------
// The depth-scaled residual operand b = bf16(x / s), s = fp32(sqrt(n)), for a BF16 value x.
//
// With y = RN(1/s), the single product RN(x y) is not always the IEEE quotient RN(x / s), but
// after the rounding to BF16 the two agree for every BF16 significand at most residual indices
// (n = 810 and 3240 are the only exceptions up to 4096).  Whether they do for a given n is a
// finite check over the 128 BF16 significands of [1, 2) (residual_mul_exact), and it carries over
// to every x = M 2^E whose product and quotient are normal FP32 numbers, because scaling by a
// power of two commutes with both roundings there.  That is the case when the biased exponent of
// x is at least residual_floor_exp(s); zero, subnormal and tiny x fall below it.  The kernels
// multiply where both conditions hold and divide (IEEE) elsewhere.  inf * y = inf / s, and NaN
// stays NaN either way.
// ---------------------------------------------------------------------------------------------

// BF16 bits of v, round to nearest even (NaN stays NaN) -- host side.
inline uint32_t bf16_bits_host(float v)
{
    uint32_t u;
    std::memcpy(&u, &v, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)
        return (u >> 16) | 0x40u;
    return (u + 0x7fffu + ((u >> 16) & 1u)) >> 16;
}

// True when bf16(RN(m y)) == bf16(RN(m / s)) for every BF16 significand m in [1, 2) (and, as a
// margin, in [2, 4)).
inline bool residual_mul_exact(float s, float y)
{
    for (int k = 128; k < 512; ++k) {
        const float m = (float)k / 128.0f;  // exact
        if (bf16_bits_host(m * y) != bf16_bits_host(m / s))
            return false;
    }
    return true;
}

// Smallest biased FP32 exponent e such that every |x| >= 2^(e - 127) has a normal product x y
// and quotient x / s: e = 1 + c with 2^c >= 2 s.
inline uint32_t residual_floor_exp(float s)
{
    uint32_t c = 0;
    while (std::ldexp(1.0f, (int)c) < 2.0f * s)
        ++c;
    return 1u + c;
}

// The kernels' rule for one BF16 value x (given as FP32), as a host reference: b as FP32.
inline float residual_operand_host(float x, float s, float y, bool mul_ok, uint32_t floor_exp)
{
    uint32_t u;
    std::memcpy(&u, &x, sizeof u);
    const uint32_t e = (u >> 23) & 0xffu;
    const uint32_t b = bf16_bits_host(mul_ok && e >= floor_exp ? x * y : x / s) << 16;
    float r;
    std::memcpy(&r, &b, sizeof r);
    return r;
}

#if defined(__CUDACC__)

typedef unsigned long long f2;  // two FP32 lanes: low = element 2i, high = element 2i+1

__device__ __forceinline__ f2 make_f2(float lo, float hi)
{
    f2 r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ f2 splat(float v) { return make_f2(v, v); }

__device__ __forceinline__ float lo_of(f2 v) { return __uint_as_float((uint32_t)v); }

__device__ __forceinline__ float hi_of(f2 v) { return __uint_as_float((uint32_t)(v >> 32)); }

__device__ __forceinline__ f2 add2(f2 a, f2 b)
{
    f2 d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2 sub2(f2 a, f2 b)
{
    f2 d;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2 mul2(f2 a, f2 b)
{
    f2 d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ f2 fma2(f2 a, f2 b, f2 c)
{
    f2 d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// BF16 pair word -> FP32 pair (exact widening)
__device__ __forceinline__ f2 widen(uint32_t w)
{
    return make_f2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// FP32 pair -> BF16 pair word, round to nearest even (NaN preserved)
__device__ __forceinline__ uint32_t narrow(f2 v)
{
    uint32_t d;
    asm("{\n\t.reg .f32 lo, hi;\n\tmov.b64 {lo, hi}, %1;\n\t"
        "cvt.rn.bf16x2.f32 %0, hi, lo;\n\t}"
        : "=r"(d)
        : "l"(v));
    return d;
}

// bf16(float(a) + float(b)) for two BF16 pairs, as one packed BF16 add.  For two BF16 operands
// the FP32 sum is exact unless their exponents differ by 16 or more, and then the smaller one is
// far below half a BF16 ulp of the larger, so rounding the FP32 sum to BF16 and rounding the
// exact sum to BF16 give the same value: the correctly rounded BF16 sum that add.rn.bf16x2
// returns.
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Packed compensated sum: two independent accumulators (hi, lo), one per lane.
struct Sum2x2 {
    f2 hi, lo;
};

// Adds t >= 0 to an accumulator with Knuth's TwoSum (an error-free transformation: the new
// hi + the new error term is exactly hi + t), the error added to lo.  (Folding a square t = x x
// into FMAs here measured 2% slower in the MoE ring.)
__device__ __forceinline__ void sum2_add(Sum2x2 &a, f2 t)
{
    const f2 s = add2(a.hi, t);
    const f2 bp = sub2(s, a.hi);
    const f2 ap = sub2(s, bp);
    const f2 e = add2(sub2(a.hi, ap), sub2(t, bp));
    a.hi = s;
    a.lo = add2(a.lo, e);
}

// Adds t = x x (exact) to an accumulator whose running sum is at least t (both lanes) with
// Dekker's Fast2Sum (s = hi + t; error t - (s - hi), exact under that condition), the square
// folded into two FMAs: s = RN(x x + hi), and the error RN(x x + (hi - s)), where hi - s is the
// exact, negated s - hi of Fast2Sum.
__device__ __forceinline__ void fast2_add_sq(Sum2x2 &a, f2 x)
{
    const f2 s = fma2(x, x, a.hi);
    const f2 e = fma2(x, x, sub2(a.hi, s));
    a.hi = s;
    a.lo = add2(a.lo, e);
}

// Merge of two packed accumulators (TwoSum of the hi parts, error added to the lo parts).
__device__ __forceinline__ Sum2x2 sum2_merge(const Sum2x2 &a, const Sum2x2 &b)
{
    const f2 s = add2(a.hi, b.hi);
    const f2 bp = sub2(s, a.hi);
    const f2 ap = sub2(s, bp);
    const f2 e = add2(sub2(a.hi, ap), sub2(b.hi, bp));
    return Sum2x2{s, add2(add2(a.lo, b.lo), e)};
}

// Lane-wise unsigned maximum of two pairs of 16-bit values.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Bit 15 of each 16-bit half stays set only if that BF16 element of `w` has an exponent field
// >= f, where floor_bits = (f << 7) | (f << 23) (a borrow trick on each half; the halves cannot
// borrow from each other because each starts at 0x8000 or more).  AND the results of several
// words and test them with exp_floor_ok().
__device__ __forceinline__ uint32_t exp_floor_bits(uint32_t w, uint32_t floor_bits)
{
    return ((w & 0x7f807f80u) | 0x80008000u) - floor_bits;
}

__device__ __forceinline__ bool exp_floor_ok(uint32_t all)
{
    return (all & 0x80008000u) == 0x80008000u;
}

#endif  // __CUDACC__

}  // namespace beam
