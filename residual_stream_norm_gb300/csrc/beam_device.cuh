// beam_device.cuh -- device helpers shared by the Beam boundary-path kernels (sm_103a).
//
// All rounding-sensitive arithmetic uses the explicit IEEE round-to-nearest intrinsics
// (__fadd_rn, __fmul_rn, ...) so that no multiply-add contraction or reassociation can change
// a result; the library is also compiled with -fmad=false.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace beam {

// ---------------------------------------------------------------------------------------------
// BF16 <-> FP32.  A 32-bit word holds two BF16 values: element 2i in the low half, 2i+1 high.
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round two FP32 values to BF16 (IEEE round-to-nearest-even, NaN preserved) and pack them.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    uint32_t d;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
    return d;
}

// ---------------------------------------------------------------------------------------------
// Global memory access.  16-byte vectors.  Streamed tensors bypass L1 allocation and use the
// coherent path (an output may be the same buffer as an input); small tensors that are
// read-only for the whole kernel (norm weights) use the default L1-cached path -- the
// non-coherent path cost a one-row (decode) boundary 0.14 us more, all of it latency.  The
// loads are volatile so that they are never moved past a store of the same kernel.
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ld_cached(const void *p)
{
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// Coherent load, for data this kernel may also write (in-place Q/K rows, in-place gate).
__device__ __forceinline__ uint4 ld_plain(const void *p)
{
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_global(void *p, uint4 v)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ float4 ld_stream_f4(const float *p)
{
    const uint4 v = ld_stream(p);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z),
                       __uint_as_float(v.w));
}

__device__ __forceinline__ void st_global_v2(void *p, uint32_t a, uint32_t b)
{
    asm volatile("st.global.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(a), "r"(b) : "memory");
}

__device__ __forceinline__ uint32_t &word(uint4 &v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

__device__ __forceinline__ uint32_t word(const uint4 &v, int i)
{
    return i == 0 ? v.x : (i == 1 ? v.y : (i == 2 ? v.z : v.w));
}

// ---------------------------------------------------------------------------------------------
// Compensated sum of non-negative FP32 terms.
//
// (hi, lo) carries a running sum whose rounding errors are captured exactly by Knuth's TwoSum
// (an error-free transformation: s + e == a + b exactly).  The final hi + lo is the FP32
// rounding of a value within ~n * 2^-48 relative of the exact sum, so the rounded result is
// the correctly rounded sum except in vanishingly rare near-tie cases -- the summation order
// (thread, warp, block) no longer decides the FP32 result.
// ---------------------------------------------------------------------------------------------

struct Sum2 {
    float hi, lo;
};

__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e)
{
    s = __fadd_rn(a, b);
    float bp = __fsub_rn(s, a);
    float ap = __fsub_rn(s, bp);
    e = __fadd_rn(__fsub_rn(a, ap), __fsub_rn(b, bp));
}

// Commutative merge: merge(a, b) and merge(b, a) give identical bits (TwoSum's error term is
// the unique exact remainder), so butterfly shuffles leave every lane with the same value.  The
// pair is not renormalised: lo gathers the exact TwoSum errors and the incoming lo terms, so after
// L merges |lo| stays within about L/2 ulp(hi), and each of its additions errs by at most
// 2^-24 |lo| -- far below the 2^-37 budget of near_tie() -- while the dependent chain per merge
// stays short.  A non-finite hi propagates as in IEEE addition (lo then becomes NaN and is
// ignored by sum_value()).
__device__ __forceinline__ Sum2 sum_merge(Sum2 a, Sum2 b)
{
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    return Sum2{s, __fadd_rn(__fadd_rn(a.lo, b.lo), e)};
}

// FP32 value of the sum.  Once hi has overflowed (or a term was inf / NaN) the error term is
// meaningless (inf - inf); hi alone then carries the IEEE result.
__device__ __forceinline__ float sum_value(Sum2 a)
{
    return isfinite(a.hi) ? __fadd_rn(a.hi, a.lo) : a.hi;
}

__device__ __forceinline__ Sum2 warp_sum(Sum2 a, int width = 32)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        if (off < width) {
            Sum2 o;
            o.hi = __shfl_xor_sync(0xffffffffu, a.hi, off);
            o.lo = __shfl_xor_sync(0xffffffffu, a.lo, off);
            a = sum_merge(a, o);
        }
    }
    return a;
}

// ---------------------------------------------------------------------------------------------
// Exact rounding of a row sum.
//
// The compensated sums above are within 2^-37 relative of the exact sum of their (non-negative,
// exactly computed) terms: an accumulator of m terms errs by at most m^2/2 u^2 (u = 2^-24; a
// thread splits its n <= 64 terms over two accumulators, n^2/4 u^2 <= 2^-38) and each of at most
// ten merge levels by about 5 u^2 more.  An accumulator seeded with an upper bound M <= S of its
// terms (S the sum of all the thread's terms; Fast2Sum in place of TwoSum, M taken off afterwards
// by an exact TwoSum) keeps its running sum below 2S, so its m error terms add up with an error
// of at most 2 m^2 u^2 S: 2^-39 S for the 16 terms of each of a RoPE lane's two accumulators.  RN(hi + lo) is the FP32 rounding of the exact sum unless
// hi + lo lies within that distance of a rounding boundary; near_tie() detects those sums
// (about 2^-12 of them) so that they can be recomputed exactly in integer arithmetic
// (beam_exact.cuh).
// ---------------------------------------------------------------------------------------------

// True when RN(hi + lo) = r1 might not be the rounding of the exact sum.
__device__ __forceinline__ bool near_tie(float hi, float lo, float r1)
{
    if (!(r1 > 0.0f) || !isfinite(r1))
        return false;  // zero (all terms zero) or non-finite: nothing to decide
    const uint32_t u = __float_as_uint(r1);
    const uint32_t e = u >> 23;
    if (e < 40u)
        return true;  // tiny sums always take the exact path
    const float half_up = __uint_as_float((e - 24u) << 23);  // ulp(r1) / 2
    const float half_dn = (u & 0x7fffffu) ? half_up : __uint_as_float((e - 25u) << 23);
    const float band = __uint_as_float((e - 36u) << 23);     // >= 2^-37 r1
    const float res = __fadd_rn(__fsub_rn(hi, r1), lo);     // hi - r1 is exact
    return res > __fsub_rn(half_up, band) || res < __fsub_rn(band, half_dn);
}

// ---------------------------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel lets the next kernel of its stream be scheduled
// as soon as it starts (launch_dependents), and reads nothing but model parameters (norm
// weights, gate bias) before griddepcontrol.wait, which returns once the preceding kernel has
// completed and its writes are visible.  Without a programmatic launch both are no-ops.
// ---------------------------------------------------------------------------------------------

__device__ __forceinline__ void pdl_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_wait()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// r = 1 / sqrt(ms / len + eps) with IEEE division and square root.  The reciprocal is the
// correctly rounded __frcp_rn: the same value as the division 1 / x.
__device__ __forceinline__ float rms_inv(float ms, float len, float eps)
{
    return __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(ms, len), eps)));
}

// The same for a power-of-two length with inv_len = 1 / len (exact): ms / len and ms * inv_len
// are the correct roundings of the same real number, so they are equal.
__device__ __forceinline__ float rms_inv_pow2(float ms, float inv_len, float eps)
{
    return __frcp_rn(__fsqrt_rn(__fadd_rn(__fmul_rn(ms, inv_len), eps)));
}

}  // namespace beam
