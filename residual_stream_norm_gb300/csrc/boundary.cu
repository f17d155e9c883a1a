// boundary.cu -- fused sublayer-boundary kernels (sm_103a).
//
// Pages cited (titles as printed):
//   [vLLM]  "Serving Reflection Beam auf vLLM ab Tag 0"
//   [SGL]   "SGLang 支撑编程模型 Beam 生产部署"
//
// One pass over each token row: post-RMSNorm of the sublayer output, the depth-scaled residual
// add with both operands rounded to BF16, and the next sublayer's pre-RMSNorm ([vLLM]
// "Agentengetriebene Optimierung" change 1; [vLLM] "MoE und Residual-Stream", bullets
// "Sandwich-Norm" and "Tiefenskalierte Residuen"; [SGL] "三明治归一化与深度缩放残差").  The MoE
// variant first forms the top-K weighted expert sum ([vLLM] change 3; [SGL] "稠密层与分组 MoE
// 路由"); the tensor-parallel variant first sums the P ranks' partial sublayer outputs (the TP
// all-reduce that [vLLM] change 3 runs inside the norm kernel, and the [SGL] kernel-fusion
// paragraph fuses with the norms and the scaled add).  Nothing between the stages goes back to
// HBM: per row the kernel reads x (or the K expert rows, or the P partial rows) and h once and
// writes h' and y once; the norm weights come from L1/L2 (rows kernel) or are parked once per
// CTA in shared memory (persistent kernels).
//
// Three layouts, same arithmetic (boundary_chain):
//  * rows kernel (few tokens, e.g. batch-1 decode): one CTA per token row; each thread owns VPT
//    16-byte vectors at vector indices tid + i * blockDim.x and loads them straight from memory.
//  * prefetch kernel (many tokens, plain boundary): a persistent grid of 4-warp CTAs, each with
//    two row buffers in shared memory that one of its threads refills with bulk TMA copies
//    (cp.async.bulk, completion on an mbarrier) two rows ahead, right after the first block
//    reduction of the row that leaves the buffer.
//  * ring kernel (many tokens, MoE and tensor-parallel variants): a persistent grid with warp
//    specialisation: one producer warp issues bulk TMA copies of each row's inputs in chunks of
//    128 vectors -- the K expert (or P partial) chunks and the h chunk -- into a ring of
//    shared-memory stages, and four consumer warps reduce and finish the rows, releasing each
//    stage on an "empty" mbarrier as soon as they have read it.
// A persistent kernel whose wait on its own copies runs out of time (kernel argument wait_ns)
// raises the device fault word and from then on writes nothing: no row computed from a buffer
// that may not have filled reaches h', y or rstd.
// Only 4 warps share a row, so the two block reductions per row stay cheap, and several CTAs fit
// on an SM.
// The row stays in registers as packed BF16 between the two block reductions; element math runs
// on packed FP32 pairs (beam_f32x2.cuh) with the same IEEE roundings as the scalar definition.

#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "beam_device.cuh"
#include "beam_exact.cuh"
#include "beam_f32x2.cuh"
#include "beam_kernels.h"
#include "beam_tma.cuh"

namespace beam {

// Fault word of this library on each device; bits are kFault* values (beam_tma.cuh).
__device__ unsigned int g_fault_word = 0u;

namespace {

constexpr int kMaxK = 16;
constexpr int kRingMaxK = 8;  // the ring takes at most 8 source slots (MoE coefficients in registers)

// Shared-memory slot of one warp in the rare exact path (beam_exact.cuh).
struct ExactSlot {
    uint64_t hi, lo;
    uint32_t sticky, max_bits;
};

// Barrier of the threads that share a row: the whole CTA (bar 0), or the `nt` threads of named
// barrier `bar` (the ring kernel's consumer warps).
__device__ __forceinline__ void group_sync(int bar, int nt)
{
    if (bar == 0)
        __syncthreads();
    else
        named_sync(bar, nt);
}

// A thread's VPT packed BF16 vectors, copied for the rare exact path.
template <int VPT>
struct Vecs {
    uint4 v[VPT];
};

// The rare exact path of block_sum_sq: the block's sum of the FP32 squares of the threads'
// vectors in 128-bit fixed point, rounded once to FP32 (beam_exact.cuh).  The largest square of
// the block sets the scale; integer sums are associative, so every thread gets the same bits.
// The vectors arrive as a copy, and the loop over them stays rolled: the rare path costs little
// code and few registers.
template <int VPT>
__device__ __forceinline__ float block_sum_exact(const Vecs<VPT> vv, ExactSlot *xslot, int nt,
                                                 int bar)
{
    const uint4 (&v)[VPT] = vv.v;
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nw = nt >> 5;
    uint32_t mx = 0;  // bits of the largest square (NaN patterns above +inf)
#pragma unroll 1
    for (int i = 0; i < VPT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const f2 x = widen(word(v[i], j));
            const uint32_t a0 = __float_as_uint(__fmul_rn(lo_of(x), lo_of(x))) & 0x7fffffffu;
            const uint32_t a1 = __float_as_uint(__fmul_rn(hi_of(x), hi_of(x))) & 0x7fffffffu;
            mx = max(mx, max(a0, a1));
        }
    mx = __reduce_max_sync(0xffffffffu, mx);
    if (lane == 0)
        xslot[warp].max_bits = mx;
    group_sync(bar, nt);
    for (int w = 0; w < nw; ++w)
        mx = max(mx, xslot[w].max_bits);
    if (mx >= 0x7f800000u)  // a NaN or infinite square: the IEEE sum
        return __uint_as_float(mx > 0x7f800000u ? 0x7fc00000u : 0x7f800000u);
    if (mx == 0u)
        return 0.0f;
    const uint32_t emax = exact_emax(mx);
    ExactAcc acc = {0ull, 0ull, 0u};
#pragma unroll 1
    for (int i = 0; i < VPT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const f2 x = widen(word(v[i], j));
            exact_add(acc, __float_as_uint(__fmul_rn(lo_of(x), lo_of(x))), emax);
            exact_add(acc, __float_as_uint(__fmul_rn(hi_of(x), hi_of(x))), emax);
        }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ExactAcc o;
        o.hi = __shfl_xor_sync(0xffffffffu, acc.hi, off);
        o.lo = __shfl_xor_sync(0xffffffffu, acc.lo, off);
        o.sticky = __shfl_xor_sync(0xffffffffu, acc.sticky, off);
        exact_merge(acc, o);
    }
    if (lane == 0) {
        xslot[warp].hi = acc.hi;
        xslot[warp].lo = acc.lo;
        xslot[warp].sticky = acc.sticky;
    }
    group_sync(bar, nt);
    ExactAcc t = {0ull, 0ull, 0u};
    for (int w = 0; w < nw; ++w)
        exact_merge(t, ExactAcc{xslot[w].hi, xslot[w].lo, xslot[w].sticky});
    return exact_round(t, emax);
}

// Compensated sum of the squares of this thread's VPT packed BF16 vectors: four independent
// packed accumulators (one per word of a vector) keep the dependent chains short.
template <int VPT>
__device__ __forceinline__ Sum2x2 squares_sum(const uint4 (&v)[VPT])
{
    Sum2x2 acc[4] = {{0ull, 0ull}, {0ull, 0ull}, {0ull, 0ull}, {0ull, 0ull}};
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const f2 x = widen(word(v[i], j));
            sum2_add(acc[j], mul2(x, x));  // x x is exact: the square of a BF16 value
        }
    return sum2_merge(sum2_merge(acc[0], acc[1]), sum2_merge(acc[2], acc[3]));
}

__device__ __forceinline__ Sum2 lanes_merged(const Sum2x2 &a)
{
    return sum_merge(Sum2{lo_of(a.hi), lo_of(a.lo)}, Sum2{hi_of(a.hi), hi_of(a.lo)});
}

// Sum over the first `nt` threads of the CTA (a multiple of 32, synchronised by
// group_sync(bar, nt)) of the squares of their vectors `v`, of which each thread has formed the
// compensated partial sum `acc`; rounded as the exact sum would be.  Warp partials go through
// `slot` / `xslot` (>= nt / 32 entries no concurrent reduction uses); every warp combines them
// with the same butterfly, so all threads get identical bits and take the rare exact path
// together.
template <int VPT>
__device__ __forceinline__ float block_sum_sq(const Sum2x2 &acc, const uint4 (&v)[VPT],
                                              Sum2 *slot, ExactSlot *xslot, int nt, int bar)
{
    const Sum2 a = warp_sum(lanes_merged(acc));
    const int lane = threadIdx.x & 31;
    const int nw = nt >> 5;
    if (lane == 0)
        slot[threadIdx.x >> 5] = a;
    group_sync(bar, nt);
    Sum2 p = lane < nw ? slot[lane] : Sum2{0.0f, 0.0f};
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        if (off < nw) {
            Sum2 o;
            o.hi = __shfl_xor_sync(0xffffffffu, p.hi, off);
            o.lo = __shfl_xor_sync(0xffffffffu, p.lo, off);
            p = sum_merge(p, o);
        }
    }
    p.hi = __shfl_sync(0xffffffffu, p.hi, 0);
    p.lo = __shfl_sync(0xffffffffu, p.lo, 0);
    const float r1 = sum_value(p);
    if (!near_tie(p.hi, p.lo, r1))
        return r1;
    // rare: the row sum is within the compensated sum's error of an FP32 rounding boundary
    Vecs<VPT> vv;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
        vv.v[i] = v[i];
    return block_sum_exact<VPT>(vv, xslot, nt, bar);
}

// Block-wide sum over `nt` threads of the squares of their vectors, in plain FP32 and a fixed
// order (per thread, then a warp butterfly, then the warps' partials in warp order), so every
// thread gets the same bits.  Used where the result only scales a product -- y = bf16((h' r') w):
// a difference of an FP32 ulp or two in r' from the exact rounding can move y by at most one
// BF16 ulp, unlike r, whose effect reaches h' through a sum that can cancel.
template <int VPT>
__device__ __forceinline__ float block_sum_sq_plain(const uint4 (&v)[VPT], float *slot, int nt,
                                                    int bar)
{
    f2 s0 = 0ull, s1 = 0ull;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const f2 x = widen(word(v[i], j));
            if (j & 1)
                s1 = fma2(x, x, s1);
            else
                s0 = fma2(x, x, s0);
        }
    const f2 s2 = add2(s0, s1);
    float t = __fadd_rn(lo_of(s2), hi_of(s2));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
        t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, off));
    const int nw = nt >> 5;
    if ((threadIdx.x & 31) == 0)
        slot[threadIdx.x >> 5] = t;
    group_sync(bar, nt);
    t = slot[0];
    for (int w = 1; w < nw; ++w)
        t = __fadd_rn(t, slot[w]);
    return t;
}

// b = bf16(x / s) by IEEE division for one vector of BF16 values: the rare path of the residual
// operand (an element below the exponent floor, or a residual index whose product rule fails).
__device__ __forceinline__ uint4 residual_operand_ieee(uint4 xh, float s)
{
    uint4 b;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const f2 q = widen(word(xh, j));
        word(b, j) = narrow(make_f2(__fdiv_rn(lo_of(q), s), __fdiv_rn(hi_of(q), s)));
    }
    return b;
}

// Where a row's sublayer output comes from.
constexpr int kSrcPlain = 0;  // x_in [T, H]
constexpr int kSrcMoe = 1;    // the top-K combine of expert_out [T, K, H]
constexpr int kSrcTp = 2;     // the rank-order sum of the P partials TpParts::p[p] [T, H]

// The extra kernel parameter of a row source: the partials for kSrcTp, nothing otherwise.
struct NoParts {
};
template <int SRC>
using SrcParts = typename std::conditional<SRC == kSrcTp, TpParts, NoParts>::type;

__device__ __forceinline__ const void *part_ptr(const TpParts &x, int p) { return x.p[p]; }
__device__ __forceinline__ const void *part_ptr(const NoParts &, int) { return nullptr; }

// The boundary chain for one row whose inputs sit in registers: xv (x) and hv (h) hold this
// thread's vectors tid + i * nt of the row (nt threads synchronised by barrier `bar`: see
// block_sum_sq).  wpo(i) / wpr(i) give the matching weight vectors.
// `after_first_sum` runs right after the first block reduction.  `fail` (persistent kernels;
// null otherwise) is the CTA's flag that a wait on its own copies ran out.  It is read right after
// the first block reduction, whose barrier follows every thread's waits for this row (a thread
// whose wait runs out raises the flag before it reaches that barrier), and then withholds this
// row's stores and those of every later row: no output is computed from a buffer that may not
// have filled.  Read there, the load overlaps the arithmetic of the rest of the chain.
template <int VPT, bool EARLY_H, typename WPost, typename WPre, typename AfterFirstSum>
__device__ __forceinline__ void boundary_chain(const BoundaryArgs &a, int64_t row,
                                               const uint4 (&xv)[VPT], const uint4 (&hv)[VPT],
                                               WPost wpo, WPre wpr, Sum2 *red,
                                               ExactSlot *xred, float *pred, int nt, int bar,
                                               const volatile int *fail,
                                               AfterFirstSum after_first_sum)
{
    const int nvec = a.H >> 3;
    const int tid = threadIdx.x;
    const int64_t row_off = row * (int64_t)a.H;

    // ---- a1: r = 1/sqrt(mean(x^2) + eps) ---------------------------------------------------
    const float r =
        rms_inv(block_sum_sq(squares_sum(xv), xv, red, xred, nt, bar), (float)a.H, a.eps);
    const bool dead = fail != nullptr && *fail != 0;
    after_first_sum();

    // ---- a1 / a2: xhat = bf16((x r) w_post); h' = bf16(bf16(alpha h) + bf16(xhat / s)) -----
    const f2 rr = splat(r), al = splat(a.alpha), ys = splat(a.inv_s);
    const uint32_t floor_bits = a.floor_bits;
    const uint32_t mul_ok = a.mul_div ? 0xffffffffu : 0u;
    uint4 hp[VPT];
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int v = tid + i * nt;
        hp[i] = make_uint4(0u, 0u, 0u, 0u);
        if (v < nvec) {
            const uint4 w = wpo(i);
            uint4 xh, bw;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                word(xh, j) = narrow(mul2(mul2(widen(word(xv[i], j)), rr), widen(word(w, j))));
            const uint32_t ok = mul_ok & exp_floor_bits(xh.x, floor_bits) &
                                exp_floor_bits(xh.y, floor_bits) &
                                exp_floor_bits(xh.z, floor_bits) & exp_floor_bits(xh.w, floor_bits);
            if (exp_floor_ok(ok)) {  // b = bf16(x_hat y), equal to bf16(x_hat / s) here
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    word(bw, j) = narrow(mul2(widen(word(xh, j)), ys));
            } else {  // zero / tiny operands, or a residual index without the product rule
                bw = residual_operand_ieee(xh, a.s);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t aw = narrow(mul2(al, widen(word(hv[i], j))));
                word(hp[i], j) = add_bf16x2(aw, word(bw, j));  // bf16(a + b)
            }
        }
    }
    // EARLY_H: h' is final, and its stores go out ahead of the second reduction, which they
    // overlap.  At one row per kernel (decode) the kernel's last stores bound its end: 0.16 us
    // less a boundary than storing h' with y.  The persistent kernels store it with y (0.5 us
    // less at 16384 rows).  The row's h was read before either way (in-place use).  A CTA whose
    // wait gave up writes nothing; the reduction's barrier stays unconditional (threads may
    // read the flag at different times).
    char *h_out = (char *)a.h_out + 2 * row_off;
    if (EARLY_H && !dead) {
#pragma unroll
        for (int i = 0; i < VPT; ++i)
            if (tid + i * nt < nvec)
                st_global(h_out + 16 * (int64_t)(tid + i * nt), hp[i]);
    }
    const f2 rr2 = splat(rms_inv(block_sum_sq_plain(hp, pred, nt, bar), (float)a.H, a.eps));
    if (dead)
        return;

    // ---- a3: y = bf16((h' r') w_pre) --------------------------------------------------------
    char *y_out = (char *)a.y_out + 2 * row_off;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int v = tid + i * nt;
        if (v < nvec) {
            const uint4 w = wpr(i);
            uint4 yv;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                word(yv, j) = narrow(mul2(mul2(widen(word(hp[i], j)), rr2), widen(word(w, j))));
            if (!EARLY_H)
                st_global(h_out + 16 * (int64_t)v, hp[i]);
            st_global(y_out + 16 * (int64_t)v, yv);
        }
    }
    if (tid == 0 && a.rstd_out)
        reinterpret_cast<float2 *>(a.rstd_out)[row] = make_float2(r, lo_of(rr2));
}

template <bool SMEM>
__device__ __forceinline__ uint4 load_vec(const unsigned char *p)
{
    return SMEM ? *reinterpret_cast<const uint4 *>(p) : ld_stream(p);
}

// x = bf16(sum_k c_k e_k) for one 16-byte vector: one FMA per slot in slot order from +0.
// `e0` points at slot 0 of this vector; slots are `slot_bytes` apart.
template <bool SMEM>
__device__ __forceinline__ void combine_slot(f2 (&acc)[4], float ck, const unsigned char *p)
{
    const uint4 ev = load_vec<SMEM>(p);
    const f2 c2 = splat(ck);
#pragma unroll
    for (int j = 0; j < 4; ++j)
        acc[j] = fma2(c2, widen(word(ev, j)), acc[j]);
}

// c holds KC >= K coefficients (the slots past K are zero).
template <bool SMEM, int KC>
__device__ __forceinline__ uint4 combine_vec(const float (&c)[KC], int K,
                                             const unsigned char *e0, size_t slot_bytes)
{
    f2 acc[4] = {0ull, 0ull, 0ull, 0ull};
    if (K == 8) {  // Beam's top-8: fully unrolled
#pragma unroll
        for (int k = 0; k < 8; ++k)
            combine_slot<SMEM>(acc, c[k], e0 + (size_t)k * slot_bytes);
    } else {
#pragma unroll 1
        for (int k = 0; k < K; ++k) {
            float ck = c[0];
#pragma unroll
            for (int kk = 1; kk < KC; ++kk)  // register-resident select of c[k]
                ck = kk == k ? c[kk] : ck;
            combine_slot<SMEM>(acc, ck, e0 + (size_t)k * slot_bytes);
        }
    }
    uint4 x;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        word(x, j) = narrow(acc[j]);
    return x;
}

// x = bf16(((x_0 + x_1) + x_2) + ... + x_{P-1}) for one 16-byte vector: FP32 adds in rank order
// starting from rank 0's value, one BF16 rounding.  src(p) points at rank p's vector.
template <bool SMEM, typename Src>
__device__ __forceinline__ uint4 reduce_vec(int P, Src src)
{
    const uint4 v0 = load_vec<SMEM>(src(0));
    f2 acc[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
        acc[j] = widen(word(v0, j));
    if (P == 8) {  // TP8: fully unrolled, every load issued before the adds need it
#pragma unroll
        for (int p = 1; p < 8; ++p) {
            const uint4 v = load_vec<SMEM>(src(p));
#pragma unroll
            for (int j = 0; j < 4; ++j)
                acc[j] = add2(acc[j], widen(word(v, j)));
        }
    } else {
#pragma unroll 1
        for (int p = 1; p < P; ++p) {
            const uint4 v = load_vec<SMEM>(src(p));
#pragma unroll
            for (int j = 0; j < 4; ++j)
                acc[j] = add2(acc[j], widen(word(v, j)));
        }
    }
    uint4 x;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        word(x, j) = narrow(acc[j]);
    return x;
}

__device__ __forceinline__ uint4 weight_vec(const void *w, int v, int nvec)
{
    return v < nvec ? ld_cached((const char *)w + 16 * (int64_t)v) : make_uint4(0u, 0u, 0u, 0u);
}

template <int KC>
__device__ __forceinline__ void routing_coeffs(const BoundaryArgs &a, int64_t row,
                                               float (&c)[KC])
{
#pragma unroll
    for (int k = 0; k < KC; ++k)
        c[k] = k < a.K ? __fmul_rn(a.topk_w[row * a.K + k], a.routed_scaling) : 0.0f;
}

// ---- rows kernel: one CTA per row, inputs straight from memory ------------------------------

template <int VPT, int SRC>
__global__ void __launch_bounds__(VPT == 1 ? 1024 : (VPT == 8 ? 256 : 512))
    boundary_rows_kernel(const BoundaryArgs a, const __grid_constant__ SrcParts<SRC> parts)
{
    __shared__ Sum2 red[32];
    __shared__ ExactSlot xred[32];
    __shared__ float pred[32];
    const int nvec = a.H >> 3;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    pdl_launch_dependents();
    uint4 wpo[VPT], wpr[VPT];  // model parameters: fetched before waiting on the previous kernel
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        wpo[i] = weight_vec(a.w_post, tid + i * nt, nvec);
        wpr[i] = weight_vec(a.w_pre, tid + i * nt, nvec);
    }
    pdl_wait();

    for (int64_t row = blockIdx.x; row < a.T; row += gridDim.x) {
        const int64_t row_off = row * (int64_t)a.H;
        const char *h_in = (const char *)a.h_in + 2 * row_off;
        uint4 xv[VPT], hv[VPT];
        float c[kMaxK];
        if constexpr (SRC == kSrcMoe)
            routing_coeffs(a, row, c);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int v = tid + i * nt;
            if (v < nvec) {
                hv[i] = ld_stream(h_in + 16 * (int64_t)v);
                if constexpr (SRC == kSrcMoe)
                    xv[i] = combine_vec<false>(c, a.K, (const unsigned char *)a.expert_out +
                                                           2 * row_off * a.K + 16 * (int64_t)v,
                                               2 * (size_t)a.H);
                else if constexpr (SRC == kSrcTp)
                    xv[i] = reduce_vec<false>(a.P, [&](int p) {
                        return (const unsigned char *)part_ptr(parts, p) + 2 * row_off +
                               16 * (int64_t)v;
                    });
                else
                    xv[i] = ld_stream((const char *)a.x_in + 2 * row_off + 16 * (int64_t)v);
            } else {
                xv[i] = make_uint4(0u, 0u, 0u, 0u);
                hv[i] = xv[i];
            }
        }
        boundary_chain<VPT, true>(
            a, row, xv, hv, [&](int i) { return wpo[i]; }, [&](int i) { return wpr[i]; }, red,
            xred, pred, nt, 0, nullptr, [] {});
    }
}

// ---- ring kernel: persistent, warp-specialised TMA pipeline ---------------------------------
//
// A CTA has NC consumer threads (a multiple of 32) and one producer warp.  Its rows are
// blockIdx.x, blockIdx.x + gridDim.x, ...; each row is cut into VPT chunks of NC 16-byte
// vectors, and consumer thread t owns vector c * NC + t of chunk c.  A unit of work is one chunk
// of one row; its stage holds the row's KIN source chunks (K expert slots, or P partials) and its
// h chunk, each NC * 16 bytes.  Per stage two mbarriers: `full` completes when the producer's
// bulk copies have landed (transaction bytes), `empty` when all consumer warps have read the
// stage (one arrive per warp).  The producer keeps `stages` units in flight.
//
// `starve` (the diagnostic beam_selftest_persistent_timeout) arms the `full` barriers without
// issuing the copies and reads no routing weights: the consumers' first wait runs out after
// a.wait_ns, and the kernel writes nothing.

// The persistent kernels (this ring and the prefetch kernel below) let the next kernel of their
// stream be launched only once a CTA has finished its rows (griddepcontrol.launch_dependents at
// the end), not at its start as the other kernels do: a persistent grid is resident all at once,
// so an early signal let the next kernel's CTAs be placed beside it while it ran.  In the
// five-kernel prefill step that cost 41 us of 669 (boundary -> MoE boundary pairs took 540 us
// against 379, MoE boundary -> Q/K RoPE 516 against 357); each kernel alone loses about 1-2 us of
// overlap with its own next launch instead.

constexpr int kRingMaxStages = 4;
constexpr int kRingHeader = 2 * kRingMaxStages * 8;  // the full and empty mbarriers

// Ring shape of the MoE and tensor-parallel variants: their stages hold K + 1 (P + 1) slices,
// so they keep slices small (4 consumer warps) at 3 CTAs per SM.
constexpr int kRingConsumers = 128;
constexpr int kRingCtasPerSm = 3;

template <int NC, int VPT, int MINB, int SRC>
__global__ void __launch_bounds__(NC + 32, MINB)
    ring_kernel(const BoundaryArgs a, const __grid_constant__ SrcParts<SRC> parts, int stages,
                bool starve)
{
    extern __shared__ __align__(128) unsigned char dyn[];
    uint64_t *full = reinterpret_cast<uint64_t *>(dyn);
    uint64_t *empty = full + kRingMaxStages;
    unsigned char *ring = dyn + kRingHeader;
    __shared__ Sum2 red[NC / 32];  // one slot per consumer warp: 3 stages fit at 3 CTAs per SM
    __shared__ ExactSlot xred[NC / 32];
    __shared__ float pred[NC / 32];
    __shared__ int fail;
    volatile int *vfail = &fail;  // written by any thread whose wait runs out

    constexpr uint32_t kSlice = NC * 16;
    const int nvec = a.H >> 3;
    const int tid = threadIdx.x;
    const int KIN = SRC == kSrcTp ? a.P : a.K;
    const uint32_t stage_bytes = (uint32_t)(KIN + 1) * kSlice;
    // the consumer threads park their slices of w_post and w_pre here ([2][VPT][NC] vectors):
    // read from shared memory inside the chain, they cost no long-latency loads
    uint4 *wsm = reinterpret_cast<uint4 *>(ring + (size_t)stages * stage_bytes);
    const int64_t first = blockIdx.x;
    const int64_t stride = gridDim.x;
    const int64_t my_rows = first < a.T ? (a.T - first + stride - 1) / stride : 0;
    const int64_t my_units = my_rows * VPT;

    if (tid == 0) {
        for (int st = 0; st < stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], NC / 32);
        }
        fail = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (tid >= NC) {
        // ---- producer warp: one lane issues every unit's copies ------------------------------
        if (tid != NC)
            return;
        pdl_wait();
        // unit u = chunk c of row `row`, in stage st of ring pass `pass` (u = pass * stages + st);
        // all four advance incrementally (no 64-bit division in the loop)
        int64_t issued = 0, row = first;
        int st = 0, c = 0;
        uint32_t pass = 0;
        for (int64_t u = 0; u < my_units; ++u) {
            if (*vfail)
                break;  // a consumer gave up waiting: issue nothing more
            // the stage's previous use (pass - 1) must have been released by the consumers.  A
            // consumer warp releases a stage only after its wait on it succeeded, so a released
            // stage's `full` phase is complete and re-arming it is legal; after a failed wait
            // the release never comes and this wait returns false once `fail` is up.
            if (pass > 0 && !mbar_wait_or_fail(&empty[st], (pass - 1) & 1u, &fail, a.wait_ns))
                break;
            const int nv = nvec - c * NC < NC ? nvec - c * NC : NC;
            const uint32_t bytes = (uint32_t)nv * 16u;
            unsigned char *dst = ring + (size_t)st * stage_bytes;
            const size_t col = (size_t)c * kSlice;
            mbar_arrive_expect_tx(&full[st], (uint32_t)(KIN + 1) * bytes);
            if (!starve) {
#pragma unroll
                for (int k = 0; k < kRingMaxK; ++k) {  // static slot indices: no local copies
                    if (k < KIN) {
                        const char *src =
                            SRC == kSrcTp
                                ? (const char *)part_ptr(parts, k) + (size_t)row * 2 * a.H
                                : (const char *)a.expert_out + ((size_t)row * KIN + k) * 2 * a.H;
                        bulk_g2s(dst + (size_t)k * kSlice, src + col, bytes, &full[st]);
                    }
                }
                bulk_g2s(dst + (size_t)KIN * kSlice,
                         (const char *)a.h_in + (size_t)row * 2 * a.H + col, bytes, &full[st]);
                issued = u + 1;
            }
            if (++c == VPT) {
                c = 0;
                row += stride;
            }
            if (++st == stages) {
                st = 0;
                ++pass;
            }
        }
        // Before leaving, make sure none of this CTA's copies is still landing (bounded): the
        // last `stages` units issued, one per stage.
        for (int64_t u = issued - stages > 0 ? issued - stages : 0; u < issued; ++u)
            (void)mbar_wait(&full[u % stages], (uint32_t)((u / stages) & 1), a.wait_ns);
        if (*vfail)
            atomicOr(&g_fault_word, kFaultCopyTimeout);
        return;
    }

    // ---- consumer warps ----------------------------------------------------------------------
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        wsm[i * NC + tid] = weight_vec(a.w_post, tid + i * NC, nvec);
        wsm[(VPT + i) * NC + tid] = weight_vec(a.w_pre, tid + i * NC, nvec);
    }
    pdl_wait();
    const int lane = tid & 31;
    // MoE: this row's and the next row's coefficients
    float c[kRingMaxK], c_next[kRingMaxK];
#pragma unroll
    for (int k = 0; k < kRingMaxK; ++k)
        c_next[k] = 0.0f;
    if (SRC == kSrcMoe && my_rows > 0 && !starve)
        routing_coeffs(a, first, c_next);
    int st = 0;          // stage of the next unit
    uint32_t parity = 0;  // phase parity of that stage's `full` barrier for this pass
    for (int64_t i = 0; i < my_rows; ++i) {
        const int64_t row = first + i * stride;
        if constexpr (SRC == kSrcMoe) {
            // this row's coefficients were fetched during the previous row; fetch the next's
#pragma unroll
            for (int k = 0; k < kRingMaxK; ++k)
                c[k] = c_next[k];
            if (i + 1 < my_rows && !starve)
                routing_coeffs(a, row + stride, c_next);
        }
        uint4 xv[VPT], hv[VPT];
#pragma unroll
        for (int ch = 0; ch < VPT; ++ch) {
            const bool landed = mbar_wait_or_fail(&full[st], parity, &fail, a.wait_ns);
            const unsigned char *stage = ring + (size_t)st * stage_bytes;
            if (ch * NC + tid < nvec) {
                hv[ch] = *reinterpret_cast<const uint4 *>(stage + (size_t)KIN * kSlice + 16 * tid);
                if constexpr (SRC == kSrcTp)
                    xv[ch] = reduce_vec<true>(
                        KIN, [&](int p) { return stage + (size_t)p * kSlice + 16 * tid; });
                else
                    xv[ch] = combine_vec<true>(c, KIN, stage + 16 * tid, kSlice);
            } else {
                xv[ch] = make_uint4(0u, 0u, 0u, 0u);
                hv[ch] = xv[ch];
            }
            __syncwarp();
            if (lane == 0 && landed)
                mbar_arrive(&empty[st]);  // this warp is done with the stage
            if (++st == stages) {
                st = 0;
                parity ^= 1u;
            }
        }
        boundary_chain<VPT, false>(
            a, row, xv, hv, [&](int k) { return wsm[k * NC + tid]; },
            [&](int k) { return wsm[(VPT + k) * NC + tid]; }, red, xred, pred, NC, 1, vfail,
            [] {});
    }
    pdl_launch_dependents();  // only now (see the note above the ring kernel)
    if (tid == 0 && *vfail)
        atomicOr(&g_fault_word, kFaultCopyTimeout);
}

// ---- prefetch kernel: persistent, every warp a consumer ---------------------------------------
//
// The plain boundary without a producer warp: a CTA of NC = 128 threads keeps NBUF row buffers
// in shared memory (x then h, nvec vectors each), filled by two bulk copies per row with one
// "full" mbarrier per buffer.  Thread t owns vectors t + c * NC of a row.  Right after the first
// block reduction of a row -- when every thread has read the row out of its buffer, since the
// reduction's barrier follows the reads -- thread 0 refills that buffer with the row NBUF rows
// ahead, so the copies fly during the rest of the row's chain and the next rows'.  The norm
// weights are parked in shared memory too: a row buffer and the weights take 40 KB for H = 5120.
//
// Once a wait has run out (the CTA's `fail` flag), thread 0 refills nothing more, so at most one
// copy per buffer can still be in flight, and the row loop writes nothing.  A refill re-arms its
// buffer's barrier only after thread 0's own wait on that buffer succeeded (the phase is
// complete): otherwise the flag is up by then, read after the reduction's barrier.  `starve` (the
// diagnostic beam_selftest_persistent_timeout) arms the buffers' barriers without issuing the
// copies.

// Launch bound: 3 CTAs an SM, the number its shared memory allows (two row buffers and the
// weights, 60 KB for H = 5120); bounded for 4, the compiler held the kernel to fewer registers
// and it took 109.3 us at T = 16384, against 107.6.
template <int VPT, int NBUF>
__global__ void __launch_bounds__(128, 3) boundary_pf_kernel(const BoundaryArgs a, bool starve)
{
    constexpr int NC = 128;
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ __align__(8) uint64_t full[NBUF];
    __shared__ Sum2 red[32];
    __shared__ ExactSlot xred[32];
    __shared__ float pred[32];
    __shared__ int fail;
    volatile int *vfail = &fail;  // written by any thread whose wait runs out
    const int nvec = a.H >> 3;
    const int tid = threadIdx.x;
    const uint32_t tbytes = (uint32_t)nvec * 16u;                  // one tensor's row
    const size_t buf_bytes = (size_t)2 * VPT * NC * 16;           // x and h slots of a buffer
    uint4 *wsm = reinterpret_cast<uint4 *>(dyn + (size_t)NBUF * buf_bytes);  // [2][VPT][NC]
    const int64_t first = blockIdx.x;
    const int64_t stride = gridDim.x;
    const int64_t my_rows = first < a.T ? (a.T - first + stride - 1) / stride : 0;

    auto issue = [&](int64_t row, int b) {
        unsigned char *dst = dyn + (size_t)b * buf_bytes;
        mbar_arrive_expect_tx(&full[b], 2u * tbytes);
        if (!starve) {
            bulk_g2s(dst, (const char *)a.x_in + (size_t)row * 2 * a.H, tbytes, &full[b]);
            bulk_g2s(dst + (size_t)VPT * NC * 16, (const char *)a.h_in + (size_t)row * 2 * a.H,
                     tbytes, &full[b]);
        }
    };

    if (tid == 0) {
        for (int b = 0; b < NBUF; ++b)
            mbar_init(&full[b], 1);
        fail = 0;
        fence_mbar_init();
    }
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        wsm[i * NC + tid] = weight_vec(a.w_post, tid + i * NC, nvec);
        wsm[(VPT + i) * NC + tid] = weight_vec(a.w_pre, tid + i * NC, nvec);
    }
    __syncthreads();
    pdl_wait();
    if (tid == 0)
        for (int b = 0; b < NBUF && b < my_rows; ++b)
            issue(first + b * stride, b);

    // refills issued by thread 0, one per row from row 0 on (they stop for good once `fail` is
    // set), so buffer b was filled 1 + |{i < refills : i = b mod NBUF}| times
    int64_t refills = 0;
    for (int64_t i = 0; i < my_rows; ++i) {
        const int64_t row = first + i * stride;
        const int b = (int)(i % NBUF);
        (void)mbar_wait_or_fail(&full[b], (uint32_t)((i / NBUF) & 1), &fail, a.wait_ns);
        const unsigned char *buf = dyn + (size_t)b * buf_bytes;
        uint4 xv[VPT], hv[VPT];
#pragma unroll
        for (int c = 0; c < VPT; ++c) {
            const int v = tid + c * NC;
            if (v < nvec) {
                xv[c] = *reinterpret_cast<const uint4 *>(buf + 16 * v);
                hv[c] = *reinterpret_cast<const uint4 *>(buf + (size_t)VPT * NC * 16 + 16 * v);
            } else {
                xv[c] = make_uint4(0u, 0u, 0u, 0u);
                hv[c] = xv[c];
            }
        }
        const bool refill = i + NBUF < my_rows;
        boundary_chain<VPT, false>(
            a, row, xv, hv, [&](int k) { return wsm[k * NC + tid]; },
            [&](int k) { return wsm[(VPT + k) * NC + tid]; }, red, xred, pred, NC, 0, vfail,
            [&] {
                if (tid == 0 && refill && !*vfail) {
                    issue(row + NBUF * stride, b);
                    ++refills;
                }
            });
    }
    pdl_launch_dependents();  // only now (see the note above the ring kernel)
    // Every copy issued was waited for above unless a wait gave up; then make sure none is still
    // landing before the CTA leaves -- the last fill of each buffer (bounded) -- and raise the
    // fault word.
    if (tid == 0 && *vfail) {
        if (!starve)
            for (int b = 0; b < NBUF && b < my_rows; ++b) {
                const int64_t fills = 1 + (refills > b ? (refills - b + NBUF - 1) / NBUF : 0);
                (void)mbar_wait(&full[b], (uint32_t)((fills - 1) & 1), a.wait_ns);
            }
        atomicOr(&g_fault_word, kFaultCopyTimeout);
    }
}

// ---- launch ----------------------------------------------------------------------------------

int device_sms()
{
    static std::mutex mu;
    static int cached_dev = -1, cached_sms = 0;
    int dev = 0;
    cudaGetDevice(&dev);
    std::lock_guard<std::mutex> lock(mu);
    if (dev != cached_dev) {
        cudaDeviceGetAttribute(&cached_sms, cudaDevAttrMultiProcessorCount, dev);
        cached_dev = dev;
    }
    return cached_sms;
}

// Resident blocks per SM of a persistent kernel with `smem` bytes of dynamic shared memory on
// the current device.  The kernel's dynamic shared-memory limit is raised (never lowered) per
// (device, kernel), and the occupancy is cached per (device, kernel, smem), so an eager launch
// pays for neither query after the first.
cudaError_t persistent_blocks(const void *kern, int threads, size_t smem, int *per_sm)
{
    static std::mutex mu;
    static std::map<std::pair<int, const void *>, size_t> smem_set;
    static std::map<std::tuple<int, const void *, size_t>, int> blocks;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    std::lock_guard<std::mutex> lock(mu);
    const auto bk = std::make_tuple(dev, kern, smem);
    const auto it = blocks.find(bk);
    if (it != blocks.end()) {
        *per_sm = it->second;
        return cudaSuccess;
    }
    size_t &lim = smem_set[std::make_pair(dev, kern)];
    if (smem > lim) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess)
            return e;
        lim = smem;
    }
    int n = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, threads, smem);
    if (e != cudaSuccess)
        return e;
    blocks[bk] = n;
    *per_sm = n;
    return cudaSuccess;
}

template <int NC, int VPT, int MINB, int SRC>
cudaError_t launch_ring(const BoundaryArgs &a, const SrcParts<SRC> &parts, int stages,
                        size_t smem, int sms, bool starve, cudaStream_t stream)
{
    auto kern = ring_kernel<NC, VPT, MINB, SRC>;
    const int threads = NC + 32;
    int per_sm = 0;
    cudaError_t e = persistent_blocks((const void *)kern, threads, smem, &per_sm);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    const int64_t slots = (int64_t)sms * per_sm;
    const unsigned grid = (unsigned)(a.T < slots ? a.T : slots);
    e = launch_pdl(kern, dim3(grid), dim3(threads), smem, stream, a, parts, stages, starve);
    return e != cudaSuccess ? e : cudaGetLastError();
}

// Smallest vectors-per-thread whose thread count fits both `max_threads` and the rows kernel's
// launch bound for that VPT (1024 threads at VPT 1, 512 at VPT 2 and 4, 256 at VPT 8).
int pick_vpt(int nvec, int max_threads)
{
    int vpt = 1;
    for (;;) {
        const int bound = vpt == 1 ? 1024 : (vpt == 8 ? 256 : 512);
        const int cap = max_threads < bound ? max_threads : bound;
        if (vpt == 8 || (nvec + vpt - 1) / vpt <= cap)
            return vpt;
        vpt *= 2;
    }
}

inline int round_warps(int n) { return (n + 31) / 32 * 32; }

// The ring launch for rows of `chunks` chunks of NC vectors: 3 stages of KIN + 1 slices beside
// the parked weights.  For 8 slots and H = 5120 that is 74 KB a CTA, which keeps 3 CTAs on an SM
// only because the kernel's static arrays are sized for its 4 consumer warps (with a third stage
// the ring no longer runs dry while the consumers finish a row's chain: 0.93 -> 0.98).
template <int NC, int MINB, int SRC>
cudaError_t launch_ring_chunks(const BoundaryArgs &a, const SrcParts<SRC> &parts, int chunks,
                               int sms, bool starve, cudaStream_t stream)
{
    const int stages = 3;
    const int kin = SRC == kSrcTp ? a.P : a.K;
    const size_t stage = (size_t)(kin + 1) * NC * 16;
    const size_t weights = (size_t)2 * chunks * NC * 16;
    const size_t smem = kRingHeader + stages * stage + weights;
    switch (chunks) {
    case 1: return launch_ring<NC, 1, MINB, SRC>(a, parts, stages, smem, sms, starve, stream);
    case 2: return launch_ring<NC, 2, MINB, SRC>(a, parts, stages, smem, sms, starve, stream);
    case 3: return launch_ring<NC, 3, MINB, SRC>(a, parts, stages, smem, sms, starve, stream);
    case 4: return launch_ring<NC, 4, MINB, SRC>(a, parts, stages, smem, sms, starve, stream);
    case 5: return launch_ring<NC, 5, MINB, SRC>(a, parts, stages, smem, sms, starve, stream);
    case 6: return launch_ring<NC, 6, MINB, SRC>(a, parts, stages, smem, sms, starve, stream);
    case 7: return launch_ring<NC, 7, MINB, SRC>(a, parts, stages, smem, sms, starve, stream);
    default: return launch_ring<NC, 8, MINB, SRC>(a, parts, stages, smem, sms, starve, stream);
    }
}

// Row buffers of the prefetch kernel, with the weights parked in shared memory: two buffers
// and the weights (60 KB for H = 5120, 3 CTAs per SM) were the fastest of the shapes measured;
// without the weights in shared memory the long-latency weight loads inside the chain cost 15%,
// and two 4-warp row groups per CTA sharing one copy of the weights (four rows in flight per SM
// instead of three) took 117.7 us against 108.8 us at T = 16384.
constexpr int kPfBuffers = 2;

template <int VPT>
cudaError_t launch_pf_vpt(const BoundaryArgs &a, int sms, bool starve, cudaStream_t stream)
{
    auto kern = boundary_pf_kernel<VPT, kPfBuffers>;
    const size_t smem = (size_t)kPfBuffers * 2 * VPT * 128 * 16 + (size_t)2 * VPT * 128 * 16;
    int per_sm = 0;
    cudaError_t e = persistent_blocks((const void *)kern, 128, smem, &per_sm);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    const int64_t slots = (int64_t)sms * per_sm;
    const unsigned grid = (unsigned)(a.T < slots ? a.T : slots);
    e = launch_pdl(kern, dim3(grid), dim3(128), smem, stream, a, starve);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t launch_pf(const BoundaryArgs &a, int chunks, int sms, bool starve,
                      cudaStream_t stream)
{
    switch (chunks) {
    case 1: return launch_pf_vpt<1>(a, sms, starve, stream);
    case 2: return launch_pf_vpt<2>(a, sms, starve, stream);
    case 3: return launch_pf_vpt<3>(a, sms, starve, stream);
    case 4: return launch_pf_vpt<4>(a, sms, starve, stream);
    case 5: return launch_pf_vpt<5>(a, sms, starve, stream);
    case 6: return launch_pf_vpt<6>(a, sms, starve, stream);
    case 7: return launch_pf_vpt<7>(a, sms, starve, stream);
    default: return launch_pf_vpt<8>(a, sms, starve, stream);
    }
}

template <int SRC>
cudaError_t launch(const BoundaryArgs &a, const SrcParts<SRC> &parts, cudaStream_t stream)
{
    const int nvec = a.H / 8;
    const int sms = device_sms();
    // Many rows (and rows of at most 8 chunks of 128 vectors): the persistent kernels, the
    // prefetch kernel for the plain boundary and the warp-specialised TMA ring for the MoE and
    // tensor-parallel variants (at most 8 source slots a row).
    const int chunks = (nvec + 127) / 128;
    const int slots = SRC == kSrcMoe ? a.K : (SRC == kSrcTp ? a.P : 0);
    if (a.T >= 4 * (int64_t)sms && chunks <= 8 && slots <= kRingMaxK) {
        if constexpr (SRC == kSrcPlain)
            return launch_pf(a, chunks, sms, false, stream);
        else
            return launch_ring_chunks<kRingConsumers, kRingCtasPerSm, SRC>(a, parts, chunks, sms,
                                                                            false, stream);
    }
    // Few rows (or very wide rows, or more than 8 slots): one CTA per row straight from memory.
    // Blocks of at most 512 threads for few rows (320 for H = 5120, two vectors a thread: a
    // decode boundary took 2.74 us in a CUDA graph, against 3.13 us with 640 threads of one
    // vector and 3.22 us with 160 of four, before its weight loads and h' stores were moved
    // off its critical path; 2.49 us since), 256 or 320 otherwise.
    const bool small = a.T < 2 * (int64_t)sms;
    const int max_threads = small ? 512 : (SRC == kSrcPlain ? 256 : 320);
    const int vpt = pick_vpt(nvec, max_threads);
    const int threads = round_warps((nvec + vpt - 1) / vpt);
    const dim3 grid((unsigned)(a.T < (int64_t)(1 << 30) ? a.T : (int64_t)(1 << 30)));
    cudaError_t e;
    switch (vpt) {
    case 1:
        e = launch_pdl(boundary_rows_kernel<1, SRC>, grid, dim3(threads), 0, stream, a,
                       parts);
        break;
    case 2:
        e = launch_pdl(boundary_rows_kernel<2, SRC>, grid, dim3(threads), 0, stream, a,
                       parts);
        break;
    case 4:
        e = launch_pdl(boundary_rows_kernel<4, SRC>, grid, dim3(threads), 0, stream, a,
                       parts);
        break;
    default:
        e = launch_pdl(boundary_rows_kernel<8, SRC>, grid, dim3(threads), 0, stream, a,
                       parts);
        break;
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_boundary(const BoundaryArgs &a, cudaStream_t stream)
{
    return launch<kSrcPlain>(a, NoParts{}, stream);
}

cudaError_t launch_moe_boundary(const BoundaryArgs &a, cudaStream_t stream)
{
    return launch<kSrcMoe>(a, NoParts{}, stream);
}

cudaError_t launch_allreduce_boundary(const BoundaryArgs &a, const TpParts &parts,
                                      cudaStream_t stream)
{
    return launch<kSrcTp>(a, parts, stream);
}

cudaError_t launch_persistent_starved(const BoundaryArgs &a, bool moe, cudaStream_t stream)
{
    const int chunks = (a.H / 8 + 127) / 128;
    const int sms = device_sms();
    if (moe)
        return launch_ring_chunks<kRingConsumers, kRingCtasPerSm, kSrcMoe>(a, NoParts{}, chunks,
                                                                            sms, true, stream);
    return launch_pf(a, chunks, sms, true, stream);
}

namespace {

// The copy-timeout path on its own: one CTA arms an mbarrier for 16 bytes of transactions that
// no copy ever delivers, waits for it with the ring kernels' bounded wait (limit `limit_ns`),
// gives up, and raises the fault bit exactly as a ring kernel would.  Nothing is in flight when
// it returns.
__global__ void copy_timeout_selftest_kernel(unsigned long long limit_ns)
{
    __shared__ __align__(8) uint64_t bar;
    __shared__ int fail;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fail = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0)
        mbar_arrive_expect_tx(&bar, 16u);  // the arrival comes; the 16 bytes never do
    __syncthreads();
    const bool ok = mbar_wait_or_fail(&bar, 0u, &fail, limit_ns);
    __syncthreads();
    if (threadIdx.x == 0 && (!ok || fail))
        atomicOr(&g_fault_word, kFaultCopyTimeout);
}

}  // namespace

cudaError_t launch_copy_timeout_selftest(unsigned long long limit_ns, cudaStream_t stream)
{
    copy_timeout_selftest_kernel<<<1, 64, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

int device_sm_count() { return device_sms(); }

cudaError_t read_fault_word(unsigned int *value, bool clear)
{
    cudaError_t e = cudaMemcpyFromSymbol(value, g_fault_word, sizeof(unsigned int));
    if (e == cudaSuccess && clear) {
        const unsigned int zero = 0u;
        e = cudaMemcpyToSymbol(g_fault_word, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace beam
