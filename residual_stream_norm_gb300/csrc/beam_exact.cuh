// beam_exact.cuh -- exactly rounded FP32 sum of non-negative FP32 terms in integer arithmetic:
// the rare path of the row and head sums of squares.
//
// The hot path sums squares with a compensated FP32 sum and rounds it; when that sum lies too
// close to an FP32 rounding boundary to trust (near_tie() in beam_device.cuh), the kernels redo
// the sum here.  Every term t = m 2^(e - 150) (m < 2^24 its significand, e >= 1 its effective
// biased exponent) is added into a 128-bit fixed-point accumulator whose scale is set by the
// largest term of the whole sum: that term's significand occupies bits [kExactTop, kExactTop + 24),
// so up to 2^14 terms cannot overflow, and terms more than 2^kExactTop below it keep their bits
// down to the accumulator's lowest bit and raise a sticky flag for what falls below.  Integer
// addition is associative, so threads may accumulate their own terms and merge in any order and
// still agree bit for bit.  The sum is then rounded once, to nearest even, from the accumulator
// and the sticky flag -- the exact rounding whenever no term lies more than 2^kExactTop below the
// largest one, and otherwise unless the exact sum falls within 2^-98 (relative) of a rounding
// boundary.  Only the integer ALU is used: FP64 is far too slow on this part for even a rare path.
#pragma once

#include <cstdint>
#include <cstring>

#if defined(__CUDACC__)
#define BEAM_EX_HD __host__ __device__ __forceinline__
#else
#define BEAM_EX_HD inline
#endif

namespace beam {

constexpr int32_t kExactTop = 88;  // bit position of the largest term's lowest significand bit

struct ExactAcc {
    uint64_t hi, lo;  // the 128-bit fixed-point sum
    uint32_t sticky;  // nonzero when some term had bits below the accumulator's lowest bit
};

BEAM_EX_HD uint32_t exact_clz64(uint64_t v)
{
#if defined(__CUDA_ARCH__)
    return (uint32_t)__clzll((long long)v);
#else
    uint32_t n = 0;
    if (v == 0)
        return 64;
    while (!(v & (1ull << 63))) {
        v <<= 1;
        ++n;
    }
    return n;
#endif
}

// Effective biased exponent of the largest term, given the largest term's bits (finite, > 0).
BEAM_EX_HD uint32_t exact_emax(uint32_t max_bits)
{
    const uint32_t e = max_bits >> 23;
    return e ? e : 1u;
}

// Adds the finite non-negative FP32 term with bits `tb`; `emax` = exact_emax() of the whole sum.
BEAM_EX_HD void exact_add(ExactAcc &a, uint32_t tb, uint32_t emax)
{
    const uint32_t e = tb >> 23;
    const uint64_t m = (uint64_t)((tb & 0x7fffffu) | (e ? 0x800000u : 0u));
    const int32_t p = kExactTop - (int32_t)emax + (int32_t)(e ? e : 1u);  // <= kExactTop
    uint64_t lo_add = 0, hi_add = 0;
    if (p >= 64) {
        hi_add = m << (p - 64);
    } else if (p >= 0) {
        lo_add = m << p;
        hi_add = p > 40 ? m >> (64 - p) : 0;
    } else if (p > -24) {
        lo_add = m >> (-p);
        a.sticky |= (uint32_t)((m & ((1ull << (-p)) - 1)) != 0);
    } else {
        a.sticky |= (uint32_t)(m != 0);
    }
    a.lo += lo_add;
    a.hi += hi_add + (a.lo < lo_add ? 1u : 0u);
}

BEAM_EX_HD void exact_merge(ExactAcc &a, const ExactAcc &b)
{
    a.lo += b.lo;
    a.hi += b.hi + (a.lo < b.lo ? 1u : 0u);
    a.sticky |= b.sticky;
}

// Bit i (0 <= i < 128) of the accumulator, and whether any bit below i is set.
BEAM_EX_HD uint32_t exact_bit(const ExactAcc &a, int32_t i)
{
    return (uint32_t)((i >= 64 ? a.hi >> (i - 64) : a.lo >> i) & 1u);
}

BEAM_EX_HD bool exact_any_below(const ExactAcc &a, int32_t i)
{
    if (i <= 0)
        return false;
    if (i >= 64)
        return a.lo != 0 || (i > 64 && (a.hi & ((1ull << (i - 64)) - 1)) != 0);
    return (a.lo & ((1ull << i) - 1)) != 0;
}

// The sum rounded to FP32, nearest even (+inf past the FP32 range).  The accumulator holds at
// least the largest term (> 0).
BEAM_EX_HD float exact_round(const ExactAcc &a, uint32_t emax)
{
    const int32_t top = a.hi ? 127 - (int32_t)exact_clz64(a.hi) : 63 - (int32_t)exact_clz64(a.lo);
    // bit 0 of the accumulator weighs 2^s, s = emax - 150 - kExactTop; the result's lowest
    // significand bit sits at bit q: 24 bits below the top, or at 2^-149 for a subnormal result
    const int32_t s = (int32_t)emax - 150 - kExactTop;
    const int32_t q_norm = top - 23, q_sub = -149 - s;
    // q >= kExactTop >= 64: a normal largest term puts top at kExactTop + 23 or above, and a
    // subnormal one (emax = 1) gives q_sub = kExactTop
    const int32_t q = q_norm > q_sub ? q_norm : q_sub;
    uint64_t keep = a.hi >> (q - 64);  // < 2^24
    const uint32_t round = exact_bit(a, q - 1);
    const bool rest = exact_any_below(a, q - 1) || a.sticky;
    if (round && (rest || (keep & 1u)))
        ++keep;
    int32_t eb = q + s + 150;  // biased exponent belonging to a significand keep in [2^23, 2^24)
    if (keep >> 24) {
        keep >>= 1;
        ++eb;
    }
    // keep < 2^23 only for a subnormal result (eb == 1); the formula covers both cases
    const uint32_t bits = eb >= 255 ? 0x7f800000u : ((uint32_t)(eb - 1) << 23) + (uint32_t)keep;
#if defined(__CUDA_ARCH__)
    return __uint_as_float(bits);
#else
    float f;
    std::memcpy(&f, &bits, sizeof f);
    return f;
#endif
}

}  // namespace beam
