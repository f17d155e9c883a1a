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
// Q/K layout: each 16-lane half-warp owns one head of 128 elements at a time, 8 per lane (lane l
// holds elements 8l..8l+7), so the rotation partner of element i (i + 64) sits in lane l ^ 8 of
// the same half-warp.  A CTA of 256 threads (16 half-warps) takes tiles of TT tokens; its work
// items are the (token, head) pairs of the tile, seven per half-warp per pass, and all loads of
// a pass are issued before any arithmetic.  The per-token factors (64 cos/sin pairs, or the
// SSMax scale) are computed once per token into shared memory while the first loads are in
// flight.  cos/sin are the FP32 roundings of the exact values of the FP32 angle
// (beam_sincos.cuh), so the rotation matches the oracle bit for bit even where its two products
// nearly cancel.  Element arithmetic runs on packed FP32 pairs (beam_f32x2.cuh).

#include "beam_device.cuh"
#include "beam_f32x2.cuh"
#include "beam_kernels.h"
#include "beam_sincos.cuh"

namespace beam {
namespace {

constexpr int kHeadDim = 128;
constexpr int kHalf = kHeadDim / 2;
constexpr int kIPP = 7;           // items per half-warp per pass (2 tokens x 56 heads = 112)
constexpr int kQkThreads = 256;   // 16 half-warps

struct RopeTable {
    float inv_freq[kHalf];  // fp32(theta^(-2i/128)), formed on the host in double
};

template <bool ROPE, int TT>
__global__ void __launch_bounds__(kQkThreads) qk_norm_kernel(const QkArgs a, const RopeTable tab)
{
    // per-token factors, double-buffered by tile parity so one barrier per tile suffices
    __shared__ __align__(16) float cs[2][TT][kHalf];
    __shared__ __align__(16) float sn[2][TT][kHalf];
    __shared__ float scale_q[2][TT];
    const int nheads = a.n_q + a.n_kv;
    const int tid = threadIdx.x;
    const int l16 = tid & 15;
    const int hw = tid >> 4;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);
    const uint4 wqv = a.n_q > 0 ? ld_cached((const char *)a.wq + 16 * l16) : zero;
    const uint4 wkv = a.n_kv > 0 ? ld_cached((const char *)a.wk + 16 * l16) : zero;
    const int64_t ntiles = (a.T + TT - 1) / TT;
    int buf = 0;

    for (int64_t tile = blockIdx.x; tile < ntiles; tile += gridDim.x, buf ^= 1) {
        const int64_t t0 = tile * TT;
        const int nt = (int)(a.T - t0 < TT ? a.T - t0 : TT);
        const int nitems = nt * nheads;

        for (int base = 0; base < nitems; base += 16 * kIPP) {
            // ---- issue the loads of this pass ------------------------------------------------
            uint4 v[kIPP];
            char *row[kIPP];
#pragma unroll
            for (int m = 0; m < kIPP; ++m) {
                const int j = base + hw + 16 * m;
                row[m] = nullptr;
                v[m] = zero;
                if (j < nitems) {
                    const int tt = j / nheads, hd = j - tt * nheads;
                    const int64_t t = t0 + tt;
                    row[m] = hd < a.n_q
                                 ? (char *)a.q + 2 * (t * a.q_stride + (int64_t)hd * kHeadDim)
                                 : (char *)a.k +
                                       2 * (t * a.k_stride + (int64_t)(hd - a.n_q) * kHeadDim);
                    v[m] = ld_plain(row[m] + 16 * l16);
                }
            }
            // ---- per-token factors of the tile, once, while the first loads fly -------------
            if (base == 0) {
                if constexpr (ROPE) {
                    for (int i = tid; i < nt * kHalf; i += kQkThreads) {
                        const int tt = i / kHalf, f = i - tt * kHalf;
                        const float p = (float)a.pos[t0 + tt];
                        const float ang = __fmul_rn(p, tab.inv_freq[f]);
                        float sv, cv;
                        if (fabsf(ang) < kSinCosMaxArg)
                            sincos_rounded(ang, &sv, &cv);  // FP32 rounding of exact cos / sin
                        else
                            sincosf(ang, &sv, &cv);
                        cs[buf][tt][f] = cv;
                        sn[buf][tt][f] = sv;
                    }
                } else {
                    if (tid < nt) {
                        const float p1 = (float)(a.pos[t0 + tid] + 1);
                        const float b = __fadd_rn(1.0f, __fdiv_rn(p1, a.ssmax_base));
                        scale_q[buf][tid] = powf(b, a.ssmax_exp);
                    }
                }
                __syncthreads();
            }
            // ---- normalise, rotate / scale, round, store -----------------------------------
#pragma unroll
            for (int m = 0; m < kIPP; ++m) {
                const int j = base + hw + 16 * m;
                const bool act = j < nitems;  // uniform across each half-warp
                const int tt = act ? j / nheads : 0;
                const int hd = act ? j - tt * nheads : 0;
                const bool isq = hd < a.n_q;
                const uint4 w = isq ? wqv : wkv;
                f2 x[4];
                Sum2x2 acc = {0ull, 0ull};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    x[q] = widen(word(v[m], q));
                    sum2_add(acc, mul2(x[q], x[q]));
                }
                Sum2 tot = sum_merge(Sum2{lo_of(acc.hi), lo_of(acc.lo)},
                                     Sum2{hi_of(acc.hi), hi_of(acc.lo)});
                tot = warp_sum(tot, 16);
                const f2 rr = splat(rms_inv(sum_value(tot), (float)kHeadDim, a.eps));
                f2 qh[4];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    qh[q] = mul2(mul2(x[q], rr), widen(word(w, q)));
                f2 out[4];
                if constexpr (ROPE) {
                    const bool first_half = l16 < 8;
                    const int fb = 8 * (l16 & 7);
                    const f2 *c2 = reinterpret_cast<const f2 *>(&cs[buf][tt][fb]);
                    const f2 *s2 = reinterpret_cast<const f2 *>(&sn[buf][tt][fb]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const f2 pe = __shfl_xor_sync(0xffffffffu, qh[q], 8);
                        const f2 qc = mul2(qh[q], c2[q]);
                        const f2 ps = mul2(pe, s2[q]);
                        // first half: q_i c - q_{i+64} s;  second half: q_{i+64} c + q_i s
                        out[q] = first_half ? sub2(qc, ps) : add2(qc, ps);
                    }
                } else {
                    const f2 sc = isq ? splat(scale_q[buf][tt]) : splat(1.0f);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        out[q] = isq ? mul2(qh[q], sc) : qh[q];
                }
                if (act) {
                    uint4 o;
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        word(o, q) = narrow(out[q]);
                    st_global(row[m] + 16 * l16, o);
                }
            }
        }
    }
}

// out = bf16(attn * 1/(1 + expf(-(gate + bias_h)))).  One CTA per row, 4 vectors per thread
// per pass, all loads of a pass issued before any arithmetic; the additions, the reciprocal's
// operand and the product run on packed pairs, expf and the IEEE reciprocal per element.
__global__ void __launch_bounds__(256) attn_gate_kernel(const GateArgs a)
{
    const int vpr = (a.n_heads * a.head_dim) >> 3;
    const int vph = a.head_dim >> 3;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const f2 one = splat(1.0f);
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
                    const f2 b = splat(a.bias[v / vph]);
                    uint4 o;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const f2 z = add2(widen(word(gv[i], j)), b);
                        const f2 e = make_f2(expf(-lo_of(z)), expf(-hi_of(z)));
                        const f2 den = add2(one, e);
                        const f2 sig = make_f2(__frcp_rn(lo_of(den)), __frcp_rn(hi_of(den)));
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

template <bool ROPE>
cudaError_t launch_qk(const QkArgs &a, cudaStream_t stream)
{
    RopeTable tab;
    for (int i = 0; i < kHalf; ++i)
        tab.inv_freq[i] = ROPE ? a.inv_freq_host[i] : 0.0f;
    // Few tokens: one token per CTA spreads them over more SMs; otherwise two per CTA.
    if (a.T < 2 * 152)
        qk_norm_kernel<ROPE, 1><<<grid_for(a.T), kQkThreads, 0, stream>>>(a, tab);
    else
        qk_norm_kernel<ROPE, 2><<<grid_for((a.T + 1) / 2), kQkThreads, 0, stream>>>(a, tab);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qk_norm_rope(const QkArgs &a, cudaStream_t stream)
{
    return launch_qk<true>(a, stream);
}

cudaError_t launch_qk_norm_ssmax(const QkArgs &a, cudaStream_t stream)
{
    return launch_qk<false>(a, stream);
}

cudaError_t launch_attn_gate(const GateArgs &a, cudaStream_t stream)
{
    const int vpr = (a.n_heads * a.head_dim) / 8;
    int threads = (vpr + 3) / 4;
    threads = threads > 256 ? 256 : threads;
    threads = (threads + 31) / 32 * 32;
    attn_gate_kernel<<<grid_for(a.T), threads, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace beam
