// beam_f32x2.cuh -- packed FP32 pair arithmetic (sm_100+ add/mul/fma .f32x2) for the
// boundary-path kernels, and the residual operand division shared with the host.
//
// Each .f32x2 instruction applies the IEEE round-to-nearest FP32 operation to both lanes, so a
// packed computation gives bit-for-bit the results of the scalar one at half the instruction
// count.  A pair holds BF16 elements 2i (low lane) and 2i+1 (high lane) of one 32-bit word.
//
// Caution: the compiler fuses a packed product that feeds a packed add/sub into one packed FMA
// (the product is then not rounded), despite the .rn modifiers and even through an opaque move.
// Packed products therefore only feed packed adds where the product is exact (squares of BF16
// values); an inexact product followed by an add uses the scalar __fmul_rn / __fadd_rn
// intrinsics, which are never fused.
#pragma once

#include <cmath>
#include <cstdint>
#include <cstring>

namespace beam {

// ---------------------------------------------------------------------------------------------
// x / s for the depth-scaled residual operand b = bf16(x / s), s = fp32(sqrt(n)).
//
// Markstein's correction step (P. Markstein, IBM J. Res. Dev. 34(1), 1990; also Cornea,
// Harrison and Tang, "Scientific Computing on Itanium-based Systems", 2002): with y = RN(1/s),
// q = RN(x * y), the remainder rem = x - q * s is exact when formed by one FMA (barring
// underflow), and q' = RN(q + rem * y) is the correctly rounded quotient.  The kernels use it for
// BF16 x with |x| >= 2^-99 (exponent field >= kMarksteinMinExp) and residual index
// n <= kMarksteinMaxN -- checked exhaustively against IEEE division for every such x and n; the
// step loses the sign of -0 and, for |x| below ~2^-109, the remainder is no longer exact, so
// smaller (and zero) x use IEEE division.  An infinite x would give NaN (inf - inf); the
// kernels take the fast path only when every |w_post| < 2^120, so that
// x = bf16((x_in * r) * w_post) cannot overflow (|x_in * r| <= sqrt(H)).  NaN stays NaN.
// ---------------------------------------------------------------------------------------------

constexpr int32_t kMarksteinMaxN = 4096;
constexpr uint32_t kMarksteinMinExp = 28;   // biased exponent of 2^-99
constexpr uint32_t kWeightMaxExp = 247;     // biased exponent of 2^120

#if defined(__CUDACC__)
#define BEAM_F2_HD __host__ __device__ __forceinline__
#else
#define BEAM_F2_HD inline
#endif

BEAM_F2_HD float div_markstein(float x, float s, float y)
{
#if defined(__CUDA_ARCH__)
    const float q = __fmul_rn(x, y);
    const float rem = __fmaf_rn(q, -s, x);
    return __fmaf_rn(rem, y, q);
#else
    const float q = x * y;
    const float rem = std::fma(q, -s, x);
    return std::fma(rem, y, q);
#endif
}

// The kernels' rule for one BF16 value x (given as FP32): the correction step where it is
// exact, IEEE division elsewhere (host reference of the device code path).
inline float residual_quotient_host(float x, int32_t n, float s, float y)
{
    uint32_t u;
    std::memcpy(&u, &x, sizeof u);
    const uint32_t e = (u >> 23) & 0xffu;
    if (n <= kMarksteinMaxN && e >= kMarksteinMinExp && e < 0xffu)
        return div_markstein(x, s, y);
    return x / s;
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

// Packed compensated sum: two independent Knuth TwoSum accumulators, one per lane.
struct Sum2x2 {
    f2 hi, lo;
};

__device__ __forceinline__ void sum2_add(Sum2x2 &a, f2 t)
{
    const f2 s = add2(a.hi, t);
    const f2 bp = sub2(s, a.hi);
    const f2 ap = sub2(s, bp);
    const f2 e = add2(sub2(a.hi, ap), sub2(t, bp));
    a.hi = s;
    a.lo = add2(a.lo, e);
}

// x / s on a pair by the correction step above (y = RN(1/s), neg_s = -s, both splatted).
__device__ __forceinline__ f2 div2_markstein(f2 x, f2 neg_s, f2 y)
{
    const f2 q = mul2(x, y);
    const f2 rem = fma2(q, neg_s, x);
    return fma2(rem, y, q);
}

// Accumulates into `all` a word whose bits 15 and 31 stay set only if both BF16 lanes of `w`
// have an exponent field >= kMarksteinMinExp (a borrow trick on each 16-bit half; the halves
// cannot borrow from each other because each starts at 0x8000 or more).
__device__ __forceinline__ void exp_floor_check(uint32_t &all, uint32_t w)
{
    constexpr uint32_t kFloor = (kMarksteinMinExp << 7) | (kMarksteinMinExp << 23);
    all &= ((w & 0x7f807f80u) | 0x80008000u) - kFloor;
}

__device__ __forceinline__ bool exp_floor_ok(uint32_t all)
{
    return (all & 0x80008000u) == 0x80008000u;
}

#endif  // __CUDACC__

}  // namespace beam
