// attention.cu -- attention-side kernels of the boundary path (sm_103a).
//
// Pages cited (titles as printed):
//   [vLLM]  "Serving Reflection Beam auf vLLM ab Tag 0"
//   [SGL]   "SGLang 支撑编程模型 Beam 生产部署"
//
//  * Per-head Q/K RMSNorm fused with RoPE (sliding-window layers) or with the SSMax query scale
//    (NoPE layers): [vLLM] "Attention", bullets "Hybride Sliding-Window- und NoPE-Schichten",
//    "SSMax auf NoPE-Schichten", "GQA mit Per-Head-Q/K-Norm"; [SGL] "混合注意力与输出门控" and
//    its kernel-fusion paragraph.
//  * Sigmoid output gate: [vLLM] "Attention", bullet "Sigmoid-Output-Gate"; [SGL]
//    "混合注意力与输出门控" and the kernel-fusion paragraph (bias add, sigmoid, multiply fused).
//
// Q/K layout: each quad of lanes owns one (token, head) item of 128 elements.  A CTA of 256
// threads takes tiles of 8 (RoPE) or 4 (SSMax) tokens, one item per quad per pass.  The direct
// kernel (qk_norm_kernel) loads a pass straight into registers; the staged kernel
// (qk_stage_kernel) copies the next pass into shared memory (cp.async) while it works on this
// one.  The
// per-token factors (64 cos/sin pairs, or the SSMax scale) are computed once per token into
// shared memory.  cos/sin are the FP32 roundings of the exact values of the FP32 angle
// (beam_sincos.cuh), so the rotation matches the oracle bit for bit even where its two products
// nearly cancel.  Element arithmetic runs on packed FP32 pairs (beam_f32x2.cuh).

#include <cuda_fp8.h>

#include "beam_device.cuh"
#include "beam_exact.cuh"
#include "beam_f32x2.cuh"
#include "beam_kernels.h"
#include "beam_sincos.cuh"
#include "beam_tma.cuh"

namespace beam {
namespace {

constexpr int kHeadDim = 128;
constexpr int kHalf = kHeadDim / 2;
constexpr int kQkThreads = 256;
constexpr int kSlots = kQkThreads / 4;  // one head per quad of lanes
constexpr int kIPP = 1;                 // heads per quad per pass, loads issued together

struct RopeTable {
    float inv_freq[kHalf];  // fp32(theta^(-2i/128)), formed on the host in double
    float neg_zero;         // -0.0f, a launch parameter so that the compiler cannot see its value
};

// The rare exact path: this quad's head sum of the FP32 squares in 128-bit fixed point, rounded
// once to FP32 (beam_exact.cuh).  Called together by the lanes of `qmask` (the quad, or the whole
// warp); the shuffles stay within quads, and each quad's special cases (all zero, a NaN or
// infinite square) are selected only at the end so that every lane takes part in every shuffle.  The lane reloads its four vectors of the head
// from `row` (still the unnormalised input: the head is stored only after this), or uses zeros
// for an inactive item (row == nullptr), so the hot loop keeps no raw copy alive for it; the
// loops stay rolled, so the rare path costs little code and few registers.
__device__ __forceinline__ float head_sum_exact(const char *row, int q, unsigned qmask)
{
    uint32_t mx = 0;  // bits of the quad's largest square (NaN patterns above +inf)
#pragma unroll 1
    for (int jj = 0; jj < 4; ++jj) {
        const uint4 v = row ? ld_plain(row + 16 * (q + 4 * jj)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int pp = 0; pp < 4; ++pp) {
            const f2 x = widen(word(v, pp));
            mx = max(mx, __float_as_uint(__fmul_rn(lo_of(x), lo_of(x))) & 0x7fffffffu);
            mx = max(mx, __float_as_uint(__fmul_rn(hi_of(x), hi_of(x))) & 0x7fffffffu);
        }
    }
    mx = max(mx, __shfl_xor_sync(qmask, mx, 1));
    mx = max(mx, __shfl_xor_sync(qmask, mx, 2));
    const bool special = mx == 0u || mx >= 0x7f800000u;
    const uint32_t emax = special ? 1u : exact_emax(mx);
    ExactAcc acc = {0ull, 0ull, 0u};
    if (!special) {
#pragma unroll 1
        for (int jj = 0; jj < 4; ++jj) {
            const uint4 v = row ? ld_plain(row + 16 * (q + 4 * jj)) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                const f2 x = widen(word(v, pp));
                exact_add(acc, __float_as_uint(__fmul_rn(lo_of(x), lo_of(x))), emax);
                exact_add(acc, __float_as_uint(__fmul_rn(hi_of(x), hi_of(x))), emax);
            }
        }
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {
        ExactAcc o;
        o.hi = __shfl_xor_sync(qmask, acc.hi, off);
        o.lo = __shfl_xor_sync(qmask, acc.lo, off);
        o.sticky = __shfl_xor_sync(qmask, acc.sticky, off);
        exact_merge(acc, o);
    }
    if (special)
        return mx == 0u ? 0.0f : __uint_as_float(mx > 0x7f800000u ? 0x7fc00000u : 0x7f800000u);
    return exact_round(acc, emax);
}

// Two FP32 pairs from four consecutive floats in shared memory (16-byte aligned): one 16-byte
// load in place of two 8-byte ones.
__device__ __forceinline__ void lds_f2x2(const float *p, f2 &a, f2 &b)
{
    const float4 v = *reinterpret_cast<const float4 *>(p);
    a = make_f2(v.x, v.y);
    b = make_f2(v.z, v.w);
}

// One 8-element vector of BF16 values `o` into a KV cache at element offset `e`: the BF16 bits
// (mode 1), or FP8 E4M3 of value / scale (mode 2; round to nearest even, saturating).  The
// quotient is IEEE division, or a product by the exact reciprocal where the scale is a power of
// two (the same value).
__device__ __forceinline__ void cache_store(void *cache, int64_t e, uint4 o, int mode, float scale,
                                            float inv, bool pow2)
{
    if (mode == 1) {
        st_global((char *)cache + 2 * e, o);
        return;
    }
    uint32_t w[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const f2 x = widen(word(o, j));
        const float lo = pow2 ? __fmul_rn(lo_of(x), inv) : __fdiv_rn(lo_of(x), scale);
        const float hi = pow2 ? __fmul_rn(hi_of(x), inv) : __fdiv_rn(hi_of(x), scale);
        w[j] = (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3);
    }
    st_global_v2((char *)cache + e, w[0] | (w[1] << 16), w[2] | (w[3] << 16));
}

// A quad of lanes owns one (token, head) item of 128 elements: lane q holds the 16-byte vectors
// q + 4 k (k = 0..3) of the head, so the rotation partners (element i < 64 and i + 64, i.e.
// vectors q + 4 k and q + 4 (k + 2)) sit in the same lane, and the head's sum of squares needs a
// two-step butterfly over the quad.  With a KV cache the items also include the V heads: their
// rows go to the V cache as they are, and the K rows go to the K cache as they are stored (after
// the norm and rotation).  Quads of one warp may then take different paths, so every shuffle is
// masked to its quad.

// The per-token factors of one tile: 64 cos/sin pairs per token (RoPE), or the SSMax query
// scale, and with a KV cache the tokens' cache slots.  cos/sin are the FP32 roundings of the exact
// values of the FP32 angle.  LAST_WARP: the CTA's last warp alone forms the cos/sin (two a
// thread for a one-token tile), so that the other warps can start on their heads meanwhile.
template <bool ROPE, bool KV, int TT, bool LAST_WARP = false>
__device__ __forceinline__ void tile_factors(const QkArgs &a, const RopeTable &tab, int64_t t0,
                                             int nt, float (&cs)[TT][kHalf],
                                             float (&sn)[TT][kHalf], float (&scale_q)[TT],
                                             int64_t (&slot)[TT])
{
    const int tid = threadIdx.x;
    if (KV && tid >= blockDim.x - TT && tid - (int)(blockDim.x - TT) < nt) {
        // the tokens' cache slots (-1: padding or out of range), by the last threads
        const int tt = tid - (int)(blockDim.x - TT);
        const int64_t s = a.slot[t0 + tt];
        slot[tt] = s >= 0 && s < a.num_slots ? s : -1;
    }
    if constexpr (ROPE) {
        const int first = LAST_WARP ? (int)blockDim.x - 1 - tid : tid;  // last warp: 0..31
        const int step = LAST_WARP ? 32 : (int)blockDim.x;
        for (int i = first; i < nt * kHalf && (!LAST_WARP || first < 32); i += step) {
            const int tt = i / kHalf, f = i - tt * kHalf;
            const float p = (float)a.pos[t0 + tt];
            const float ang = __fmul_rn(p, tab.inv_freq[f]);
            float sv, cv;
            if (fabsf(ang) < kSinCosMaxArg)
                sincos_rounded(ang, &sv, &cv);  // FP32 rounding of exact cos / sin
            else
                sincosf(ang, &sv, &cv);
            cs[tt][f] = cv;
            sn[tt][f] = sv;
        }
    } else {
        if (tid < nt) {
            const float p1 = (float)(a.pos[t0 + tid] + 1);
            const float b = __fadd_rn(1.0f, __fdiv_rn(p1, a.ssmax_base));
            scale_q[tid] = powf(b, a.ssmax_exp);
        }
    }
}

// One item: normalise, rotate / scale, round, store (and write the KV cache).  `v` holds the
// lane's four vectors (see above), `row` the item's row in global memory (nullptr: an inactive
// item, whose lanes still take part in every shuffle), `hd` its head (Q heads, then K, then V),
// `tslot` its token's cache slot, `cst` / `snt` / `sq` the token's factors.  All lanes of the
// warp call it together.  `before_rotate` runs right before the rotation reads cos/sin (RoPE).
template <bool ROPE, bool KV, typename BeforeRotate>
__device__ __forceinline__ void qk_item(const QkArgs &a, const uint4 (&v)[4], char *row, int hd,
                                        int64_t tslot, int q, unsigned qmask,
                                        const float (&wsm)[2][kHeadDim], const float *cst,
                                        const float *snt, float sq, f2 nz,
                                        BeforeRotate before_rotate)
{
    const int nqk = a.n_q + a.n_kv;
    const bool act = row != nullptr;  // uniform across each quad
    const bool isq = hd < a.n_q;
    // the cache slot of a K or V item (-1: no cache, padding or out of range); tslot is the
    // token's slot, checked against the cache when the tile's factors were formed
    const int64_t cslot = KV && act && !isq ? tslot : -1;
    if (KV && hd >= nqk) {  // a V item: into the V cache, unchanged
        if (cslot >= 0) {
            const int64_t e0 = (cslot * a.n_kv + (hd - nqk)) * kHeadDim;
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                cache_store(a.v_cache, e0 + 8 * (q + 4 * jj), v[jj], a.cache_mode,
                            a.v_scale, a.v_inv, a.v_pow2);
        }
        return;
    }
    f2 x[4][4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj)
#pragma unroll
        for (int pp = 0; pp < 4; ++pp)
            x[jj][pp] = widen(word(v[jj], pp));
    float ms;
    if constexpr (ROPE) {
        // The rotation can cancel, so an FP32 ulp of r could move an output by more than a BF16
        // ulp: the head sum is rounded as the exact sum would be.
        // Each of the two packed accumulators starts from M, the largest square of the lane,
        // so that its running sum is never below the next term and Dekker's Fast2Sum (3 adds)
        // is exact in place of TwoSum (6); 2M is taken off after the lanes are merged.  The
        // lane's largest |x| comes from an integer maximum of the BF16 magnitude bits (which
        // order like the magnitudes; a NaN element gives a NaN M, and the sum then takes the
        // exact path below, as an infinite one does), off the FP32 pipe.
        uint32_t mw = 0u;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int pp = 0; pp < 4; ++pp)
                mw = max_u16x2(mw, word(v[jj], pp) & 0x7fff7fffu);
        const float mabs = __uint_as_float(max(mw & 0xffffu, mw >> 16) << 16);
        const float m2 = __fmul_rn(mabs, mabs);  // exact: the square of a BF16 value
        Sum2x2 acc = {splat(m2), 0ull};
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int pp = 0; pp < 4; ++pp)
                fast2_add_sq(acc, x[jj][pp]);
        Sum2 tot = sum_merge(Sum2{lo_of(acc.hi), lo_of(acc.lo)}, Sum2{hi_of(acc.hi), hi_of(acc.lo)});
        tot = sum_merge(tot, Sum2{-__fadd_rn(m2, m2), 0.0f});
#pragma unroll
        for (int off = 1; off < 4; off <<= 1) {
            Sum2 o;
            o.hi = __shfl_xor_sync(qmask, tot.hi, off);
            o.lo = __shfl_xor_sync(qmask, tot.lo, off);
            tot = sum_merge(tot, o);
        }
        ms = sum_value(tot);
        // the same in the quad; a non-finite sum (an infinite or NaN square, or a seeded sum
        // past the FP32 range) is decided by the exact path too
        const bool tie = near_tie(tot.hi, tot.lo, ms) || !isfinite(ms);
        if constexpr (KV) {
            if (tie)  // rare
                ms = head_sum_exact(row, q, qmask);
        } else if (__any_sync(0xffffffffu, tie)) {
            // rare; the whole warp joins the (warp-wide) shuffles
            const float exact = head_sum_exact(row, q, qmask);
            if (tie)
                ms = exact;
        }
    } else {
        // The outputs only scale with r: a plain FP32 sum in a fixed order (per lane, then the
        // quad butterfly) moves them by at most one BF16 ulp.
        f2 s0 = 0ull, s1 = 0ull;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                if (pp & 1)
                    s1 = fma2(x[jj][pp], x[jj][pp], s1);
                else
                    s0 = fma2(x[jj][pp], x[jj][pp], s0);
            }
        const f2 s2 = add2(s0, s1);
        ms = __fadd_rn(lo_of(s2), hi_of(s2));
        ms = __fadd_rn(ms, __shfl_xor_sync(qmask, ms, 1));
        ms = __fadd_rn(ms, __shfl_xor_sync(qmask, ms, 2));
    }
    const f2 rr = splat(rms_inv_pow2(ms, 1.0f / kHeadDim, a.eps));
    const float *wrow = wsm[isq ? 0 : 1];
    f2 qh[4][4];
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
        const int e0 = 8 * (q + 4 * jj);
#pragma unroll
        for (int pp = 0; pp < 4; pp += 2) {
            f2 w0, w1;
            lds_f2x2(&wrow[e0 + 2 * pp], w0, w1);
            qh[jj][pp] = mul2(mul2(x[jj][pp], rr), w0);
            qh[jj][pp + 1] = mul2(mul2(x[jj][pp + 1], rr), w1);
        }
    }
    f2 out[4][4];
    if constexpr (ROPE) {
        before_rotate();
#pragma unroll
        for (int jj = 0; jj < 2; ++jj) {
            const int i0 = 8 * (q + 4 * jj);  // first-half element index (< 64)
            f2 cc[4], ss[4];
            lds_f2x2(&cst[i0], cc[0], cc[1]);
            lds_f2x2(&cst[i0 + 4], cc[2], cc[3]);
            lds_f2x2(&snt[i0], ss[0], ss[1]);
            lds_f2x2(&snt[i0 + 4], ss[2], ss[3]);
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                const f2 c = cc[pp], sv = ss[pp];
                const f2 lo = qh[jj][pp], hi = qh[jj + 2][pp];
                // out_i = q_i c - q_{i+64} s;  out_{i+64} = q_{i+64} c + q_i s, each product
                // rounded.  A packed product that feeds a packed add is fused into one FMA by the
                // compiler, so each product is formed as fma(x, y, nz) with nz = -0 (the same
                // value as the rounded product, signed zeros included), which it cannot fuse.
                out[jj][pp] = sub2(fma2(lo, c, nz), fma2(hi, sv, nz));
                out[jj + 2][pp] = add2(fma2(hi, c, nz), fma2(lo, sv, nz));
            }
        }
    } else {
        const f2 sc = splat(isq ? sq : 1.0f);
#pragma unroll
        for (int jj = 0; jj < 4; ++jj)
#pragma unroll
            for (int pp = 0; pp < 4; ++pp)
                out[jj][pp] = isq ? mul2(qh[jj][pp], sc) : qh[jj][pp];
    }
    if (act) {
        const int64_t e0 = KV && cslot >= 0 ? (cslot * a.n_kv + (hd - a.n_q)) * kHeadDim : 0;
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
            uint4 o;
#pragma unroll
            for (int pp = 0; pp < 4; ++pp)
                word(o, pp) = narrow(out[jj][pp]);
            const int vi = q + 4 * jj;
            st_global(row + 16 * vi, o);
            if (KV && cslot >= 0)  // a K item: the stored K' also into the K cache
                cache_store(a.k_cache, e0 + 8 * vi, o, a.cache_mode, a.k_scale, a.k_inv,
                            a.k_pow2);
        }
    }
}

// m = ceil(2^32 / n), in 64 bits (2^32 itself for n = 1): with e = m n - 2^32 < n,
// floor(j m / 2^32) = floor(j / n) whenever j e < 2^32 -- for every j < 2^14 when n < 2^12 (here
// n <= 2048 heads, j < 8 n).
__device__ __forceinline__ uint64_t div_magic(int n)
{
    return ((1ull << 32) + (uint64_t)n - 1) / (uint64_t)n;
}

// Token tt and head hd of item j of a tile of items (token-major, nheads heads a token);
// inactive items (j >= nitems) map to (0, 0).
__device__ __forceinline__ void item_of(int j, int nitems, int nheads, uint64_t hmag, int &tt,
                                        int &hd)
{
    const uint32_t jj = j < nitems ? (uint32_t)j : 0u;
    tt = (int)(((uint64_t)jj * hmag) >> 32);
    hd = (int)jj - tt * nheads;
}

// Global row of item (token t, head hd): Q heads, then K, then V.
__device__ __forceinline__ char *item_row(const QkArgs &a, int64_t t, int hd, int nqk)
{
    if (hd < a.n_q)
        return (char *)a.q + 2 * (t * a.q_stride + (int64_t)hd * kHeadDim);
    if (hd < nqk)
        return (char *)a.k + 2 * (t * a.k_stride + (int64_t)(hd - a.n_q) * kHeadDim);
    return (char *)a.v + 2 * (t * a.v_stride + (int64_t)(hd - nqk) * kHeadDim);  // only read
}

// Direct kernel: a CTA of 256 threads takes tiles of TT tokens, each quad kIPP items per pass,
// all loads of a pass issued (straight from global memory) before any arithmetic; the tile's
// factors are computed while the first loads are in flight.  The Q and K norm weights are held
// in shared memory as FP32.  SPLIT (RoPE without a cache, one-token tiles): the last warp forms
// the token's cos/sin while the other warps take their heads through the norm, and the barrier
// comes right before the rotation (Beam's 56 heads leave that warp without a head).  It pays
// while every CTA is resident at once (at most 4 an SM): 5.73 against 6.34 us at T = 128, 5.42
// against 5.56 at 608; with more rounds of CTAs the wider cos/sin chain of one warp costs more
// than it hides (10.32 against 10.18 us at 1216).
template <bool ROPE, int TT, bool KV, bool SPLIT = false>
__global__ void __launch_bounds__(kQkThreads, 4) qk_norm_kernel(const QkArgs a, const RopeTable tab)
{
    __shared__ __align__(16) float cs[2][TT][kHalf];  // double-buffered by tile parity
    __shared__ __align__(16) float sn[2][TT][kHalf];
    __shared__ float scale_q[2][TT];
    __shared__ int64_t tslot[2][TT];
    __shared__ __align__(16) float wsm[2][kHeadDim];  // wq, wk as FP32
    const int nqk = a.n_q + a.n_kv;
    const int nheads = nqk + (KV ? a.n_kv : 0);  // Q, K, then V heads
    const uint64_t hmag = div_magic(nheads);
    // shuffles: masked to the quad when V items may send quads of a warp different ways,
    // warp-wide otherwise
    const unsigned qmask = KV ? 0xfu << (threadIdx.x & 28) : 0xffffffffu;
    const int tid = threadIdx.x;
    const int q = tid & 3;
    const int slot = tid >> 2;
    pdl_launch_dependents();
    {  // model parameters: fetched before waiting on the previous kernel
        const int which = tid >> 7, e = tid & 127;
        const bool have = which == 0 ? a.n_q > 0 : a.n_kv > 0;
        const uint16_t *w = (const uint16_t *)(which == 0 ? a.wq : a.wk);
        wsm[which][e] = have ? __uint_as_float((uint32_t)w[e] << 16) : 0.0f;
    }
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const int64_t ntiles = (a.T + TT - 1) / TT;
    constexpr bool kSplit = SPLIT && ROPE && !KV && TT == 1;
    int buf = 0;
    __syncthreads();
    pdl_wait();

    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, buf ^= 1) {
        const int64_t t0 = tile * TT;
        const int nt = (int)(a.T - t0 < TT ? a.T - t0 : TT);
        const int nitems = nt * nheads;

        for (int base = 0; base < nitems; base += kSlots * kIPP) {
            // ---- issue the loads of this pass ------------------------------------------------
            uint4 v[kIPP][4];
            char *row[kIPP];
            int tok[kIPP], head[kIPP];
#pragma unroll
            for (int m = 0; m < kIPP; ++m) {
                const int j = base + slot + kSlots * m;
                int tt, hd;
                item_of(j, nitems, nheads, hmag, tt, hd);
                tok[m] = tt;
                head[m] = hd;
                row[m] = j < nitems ? item_row(a, t0 + tt, hd, nqk) : nullptr;
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    v[m][jj] = row[m] ? ld_plain(row[m] + 16 * (q + 4 * jj)) : zero;
            }
            // ---- per-token factors of the tile, once, while the first loads fly (kSplit: by
            // the last warp, with the barrier before the rotation) ----------------------------
            if (base == 0) {
                tile_factors<ROPE, KV, TT, kSplit>(a, tab, t0, nt, cs[buf], sn[buf],
                                                   scale_q[buf], tslot[buf]);
                if (!kSplit)
                    __syncthreads();
            }
#pragma unroll
            for (int m = 0; m < kIPP; ++m)
                qk_item<ROPE, KV>(a, v[m], row[m], head[m], KV ? tslot[buf][tok[m]] : -1, q,
                                  qmask, wsm, cs[buf][tok[m]], sn[buf][tok[m]],
                                  ROPE ? 0.0f : scale_q[buf][tok[m]], splat(tab.neg_zero),
                                  [&] {
                                      if (kSplit && m == 0 && base == 0)
                                          __syncthreads();
                                  });
        }
    }
}

// 16-byte asynchronous copy global -> shared (cp.async, L2 only), and its group bookkeeping.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem)
                 : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

// Waits until at most one of this thread's copy groups is still pending.
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Staged kernel (many tokens): the direct kernel's tiles, one head per quad per pass, with each
// thread's four vectors of the next pass copied into shared memory (cp.async) while it works on
// this pass, so two passes' reads are in flight per thread without holding registers for them.
// A thread reads back only what it copied itself, so no barrier guards the staging buffers;
// [pass parity][vector][thread] keeps a warp's reads of one vector contiguous (no bank
// conflicts).
// 4 CTAs of 8 warps on an SM (at most 64 registers) without a KV cache; with one, 3 CTAs (at most
// 85): at 64 its V path and cache stores spilled, and it took 110.6 us against 104.8 us at
// T = 16384.
template <bool ROPE, int TT, bool KV>
__global__ void __launch_bounds__(kQkThreads, KV ? 3 : 4)
    qk_stage_kernel(const QkArgs a, const RopeTable tab)
{
    __shared__ __align__(16) float cs[2][TT][kHalf];  // double-buffered by tile parity
    __shared__ __align__(16) float sn[2][TT][kHalf];
    __shared__ float scale_q[2][TT];
    __shared__ int64_t tslot[2][TT];
    __shared__ __align__(16) float wsm[2][kHeadDim];
    __shared__ __align__(16) uint4 stage[2][4][kQkThreads];
    const int nqk = a.n_q + a.n_kv;
    const int nheads = nqk + (KV ? a.n_kv : 0);
    const uint64_t hmag = div_magic(nheads);
    const unsigned qmask = KV ? 0xfu << (threadIdx.x & 28) : 0xffffffffu;
    const int tid = threadIdx.x;
    const int q = tid & 3;
    const int slot = tid >> 2;
    pdl_launch_dependents();
    {
        const int which = tid >> 7, e = tid & 127;
        const bool have = which == 0 ? a.n_q > 0 : a.n_kv > 0;
        const uint16_t *w = (const uint16_t *)(which == 0 ? a.wq : a.wk);
        wsm[which][e] = have ? __uint_as_float((uint32_t)w[e] << 16) : 0.0f;
    }
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const int64_t ntiles = (a.T + TT - 1) / TT;
    int buf = 0;
    __syncthreads();
    pdl_wait();

    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, buf ^= 1) {
        const int64_t t0 = tile * TT;
        const int nt = (int)(a.T - t0 < TT ? a.T - t0 : TT);
        const int nitems = nt * nheads;
        const int npass = (nitems + kSlots - 1) / kSlots;
        // item of pass p for this quad: token tt and head hd of the tile, or none; located once,
        // when its copies are issued, and carried to the pass that processes it
        auto locate = [&](int p, int &tt, int &hd) -> char * {
            const int j = p * kSlots + slot;
            item_of(j, nitems, nheads, hmag, tt, hd);
            return j < nitems ? item_row(a, t0 + tt, hd, nqk) : nullptr;
        };
        auto issue = [&](int p, const char *row) {
            if (row)
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    cp_async16(&stage[p & 1][jj][tid], row + 16 * (q + 4 * jj));
            cp_async_commit();
        };
        int tt_n, hd_n;
        char *row_n = locate(0, tt_n, hd_n);
        issue(0, row_n);
        for (int p = 0; p < npass; ++p) {
            const int tt = tt_n, hd = hd_n;
            char *row = row_n;
            if (p + 1 < npass) {
                row_n = locate(p + 1, tt_n, hd_n);
                issue(p + 1, row_n);
            } else {
                cp_async_commit();  // an empty group keeps "all but the newest" meaning pass p
            }
            if (p == 0) {  // the tile's factors, while the first copies fly
                tile_factors<ROPE, KV, TT>(a, tab, t0, nt, cs[buf], sn[buf], scale_q[buf],
                                           tslot[buf]);
                __syncthreads();
            }
            cp_async_wait_one();
            uint4 v[4];
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                v[jj] = row ? stage[p & 1][jj][tid] : zero;
            qk_item<ROPE, KV>(a, v, row, hd, KV ? tslot[buf][tt] : -1, q, qmask, wsm,
                              cs[buf][tt], sn[buf][tt], ROPE ? 0.0f : scale_q[buf][tt],
                              splat(tab.neg_zero), [] {});
        }
    }
}

// Head of vector v: floor(v / vph), vph = head_dim / 8 vectors per head, as floor(v * m / 2^32)
// with m = ceil(2^32 / vph) (gate_head_magic()).  With e = m * vph - 2^32 < vph the quotient is
// exact whenever v * e < 2^32; here v < 1024 * vph and vph <= 128, so v * e < 2^24.
__device__ __forceinline__ int gate_head(int v, uint64_t m)
{
    return (int)(((uint64_t)(uint32_t)v * m) >> 32);
}

// Hardware reciprocal (rcp.approx.f32, subnormals kept): within one FP32 ulp.
__device__ __forceinline__ float rcp_approx(float x)
{
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// out = bf16(attn * 1/(1 + expf(-(gate + bias_h)))).  One CTA per row, 4 vectors per thread
// per pass, all loads of a pass issued before any arithmetic; the additions, the reciprocal's
// operand and the product run on packed pairs, expf and the reciprocal per element.  The output
// is a product of attn and the sigmoid (nothing cancels), so the few FP32 ulps of expf and of
// the hardware reciprocal move it by at most one BF16 ulp; 1/(1 + 1) = 0.5 and 1/inf = 0 stay
// exact, so a zero gate input halves attn exactly and a -inf bias switches a head off.
__global__ void __launch_bounds__(256) attn_gate_kernel(const GateArgs a)
{
    const int vpr = (a.n_heads * a.head_dim) >> 3;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const f2 one = splat(1.0f);
    pdl_launch_dependents();
    pdl_wait();
    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        const char *attn = (const char *)a.attn + 2 * t * a.attn_stride;
        const char *gate = (const char *)a.gate + 2 * t * a.gate_stride;
        char *out = (char *)a.out + 2 * t * a.out_stride;
        for (int v0 = 0; v0 < vpr; v0 += 4 * nt) {
            uint4 av[4], gv[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int v = v0 + tid + i * nt;
                if (v < vpr) {
                    av[i] = ld_stream(attn + 16 * (int64_t)v);
                    gv[i] = ld_stream(gate + 16 * (int64_t)v);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int v = v0 + tid + i * nt;
                if (v < vpr) {
                    const f2 b = splat(a.bias[gate_head(v, a.head_magic)]);
                    uint4 o;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const f2 z = add2(widen(word(gv[i], j)), b);
                        const f2 e = make_f2(expf(-lo_of(z)), expf(-hi_of(z)));
                        const f2 den = add2(one, e);
                        const f2 sig = make_f2(rcp_approx(lo_of(den)), rcp_approx(hi_of(den)));
                        word(o, j) = narrow(mul2(widen(word(av[i], j)), sig));
                    }
                    st_global(out + 16 * (int64_t)v, o);
                }
            }
        }
    }
}

inline unsigned grid_for(int64_t units)
{
    return (unsigned)(units < (int64_t)(1 << 30) ? units : (int64_t)(1 << 30));
}

template <bool ROPE, bool KV>
cudaError_t launch_qk(const QkArgs &a, cudaStream_t stream)
{
    RopeTable tab;
    for (int i = 0; i < kHalf; ++i)
        tab.inv_freq[i] = ROPE ? a.inv_freq_host[i] : 0.0f;
    tab.neg_zero = -0.0f;
    const int64_t sms = device_sm_count();
    // Tile sizes by tokens per SM, so that the CTAs come close to filling whole rounds of 4 an
    // SM (times at T tokens, each alternative timed back to back on one GB300):
    //  * Many tokens (RoPE and the KV-cache variants from 32 an SM, plain SSMax from 8): 4 CTAs
    //    of 8 warps on an SM, one head per quad per pass, tiles of 8 tokens for RoPE (each
    //    thread then forms two cos/sin pairs per tile) and 4 for SSMax.  The staged kernel keeps
    //    a second pass's reads in flight; it pays off where a head costs the most arithmetic
    //    (RoPE) or the V rows add reads (the KV cache), while plain SSMax is as fast without it.
    //    Its 8-token tiles need many tokens to fill the GPU: RoPE took 25.4 us at T = 2048 and
    //    31-33 us at 4096 with them, against 14.1 and 27.4 us on one-token tiles, and at 8192
    //    still 45.2 against 50.6 us on two-token tiles.
    //  * Up to 4 tokens an SM: one-token tiles.  RoPE without a cache then splits its cos/sin
    //    off to the last warp (5.42 against 5.96 us at T = 608 on two-token tiles).
    //  * In between: two-token tiles.  RoPE: 9.17 against 10.24 us (one-token tiles) at
    //    T = 1216, 13.07 against 14.66 at 2048; with a KV cache 10.84 against 12.07 at 1216 and
    //    28.73 against 31.38 at 4096; SSMax: 3.55 against 4.49 us (4-token tiles) at 608, 5.18
    //    against 5.77 at 1216, but 9.17 against 9.00 at 2048, where its many-token kernel
    //    starts.
    const bool many = ROPE || KV ? a.T >= 32 * sms : a.T > 8 * sms;
    constexpr int TT = ROPE ? 8 : 4;
    const dim3 block(kQkThreads);
    cudaError_t e;
    if (many) {
        const dim3 grid(grid_for((a.T + TT - 1) / TT));
        if constexpr (ROPE || KV)
            e = launch_pdl(qk_stage_kernel<ROPE, TT, KV>, grid, block, 0, stream, a, tab);
        else
            e = launch_pdl(qk_norm_kernel<ROPE, TT, KV>, grid, block, 0, stream, a, tab);
    } else if (a.T <= 4 * sms) {
        if constexpr (ROPE && !KV)
            e = launch_pdl(qk_norm_kernel<ROPE, 1, KV, true>, dim3(grid_for(a.T)), block, 0,
                           stream, a, tab);
        else
            e = launch_pdl(qk_norm_kernel<ROPE, 1, KV>, dim3(grid_for(a.T)), block, 0, stream,
                           a, tab);
    } else {
        e = launch_pdl(qk_norm_kernel<ROPE, 2, KV>, dim3(grid_for((a.T + 1) / 2)), block, 0,
                       stream, a, tab);
    }
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_norm_rope(const QkArgs &a, cudaStream_t stream)
{
    return a.cache_mode ? launch_qk<true, true>(a, stream) : launch_qk<true, false>(a, stream);
}

cudaError_t launch_qk_norm_ssmax(const QkArgs &a, cudaStream_t stream)
{
    return a.cache_mode ? launch_qk<false, true>(a, stream) : launch_qk<false, false>(a, stream);
}

uint64_t gate_head_magic(int32_t head_dim)
{
    const uint64_t vph = (uint64_t)(head_dim / 8);
    return ((1ull << 32) + vph - 1) / vph;
}

cudaError_t launch_attn_gate(const GateArgs &a, cudaStream_t stream)
{
    const int vpr = (a.n_heads * a.head_dim) / 8;
    int threads = (vpr + 3) / 4;
    threads = threads > 256 ? 256 : threads;
    threads = (threads + 31) / 32 * 32;
    const cudaError_t e =
        launch_pdl(attn_gate_kernel, dim3(grid_for(a.T)), dim3(threads), 0, stream, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace beam
