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
// Q/K layout: one CTA per token; each 16-lane half-warp owns one head of 128 elements, 8 per
// lane (lane l holds elements 8l..8l+7), so the rotation partner of element i (i + 64) sits in
// lane l ^ 8 of the same half-warp.  The per-token factors (64 cos/sin pairs, or the SSMax
// scale) are computed once per CTA into shared memory.  cos/sin are the FP32 roundings of the
// exact values of the FP32 angle (beam_sincos.cuh), so the rotation matches the oracle bit for
// bit even where its two products nearly cancel.

#include "beam_device.cuh"
#include "beam_kernels.h"
#include "beam_sincos.cuh"

namespace beam {
namespace {

constexpr int kHeadDim = 128;
constexpr int kHalf = kHeadDim / 2;

struct RopeTable {
    float inv_freq[kHalf];  // fp32(theta^(-2i/128)), formed on the host in double
};

template <bool ROPE>
__global__ void __launch_bounds__(1024) qk_norm_kernel(const QkArgs a, const RopeTable tab)
{
    __shared__ float cs[kHalf], sn[kHalf];
    __shared__ float scale_q;
    const int nheads = a.n_q + a.n_kv;
    const int tid = threadIdx.x;
    const int l16 = tid & 15;
    const int group = tid >> 4;
    const int ngroups = blockDim.x >> 4;

    for (int64_t t = blockIdx.x; t < a.T; t += gridDim.x) {
        if constexpr (ROPE) {
            const float p = (float)a.pos[t];
            for (int i = tid; i < kHalf; i += blockDim.x) {
                const float ang = __fmul_rn(p, tab.inv_freq[i]);
                float sv, cv;
                if (fabsf(ang) < kSinCosMaxArg)
                    sincos_rounded(ang, &sv, &cv);  // FP32 rounding of the exact cos / sin
                else
                    sincosf(ang, &sv, &cv);
                cs[i] = cv;
                sn[i] = sv;
            }
        } else {
            if (tid == 0) {
                const double p1 = (double)a.pos[t] + 1.0;
                scale_q = (float)pow(1.0 + p1 / (double)a.ssmax_base, (double)a.ssmax_exp);
            }
        }
        __syncthreads();

        // Uniform trip count for the whole block keeps the shuffles below converged.
        for (int hb = 0; hb < nheads; hb += ngroups) {
            const int hd = hb + group;
            const bool act = hd < nheads;
            const bool isq = hd < a.n_q;
            char *row = nullptr;
            uint4 v = make_uint4(0u, 0u, 0u, 0u), w = v;
            if (act) {
                row = isq ? (char *)a.q + 2 * (t * a.q_stride + (int64_t)hd * kHeadDim)
                          : (char *)a.k + 2 * (t * a.k_stride + (int64_t)(hd - a.n_q) * kHeadDim);
                v = ld_plain(row + 16 * l16);
                w = ld_cached((const char *)(isq ? a.wq : a.wk) + 16 * l16);
            }
            Sum2 s0 = {0.0f, 0.0f}, s1 = {0.0f, 0.0f};
            float x[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                x[2 * j] = bf_lo(word(v, j));
                x[2 * j + 1] = bf_hi(word(v, j));
                sum_add(s0, __fmul_rn(x[2 * j], x[2 * j]));
                sum_add(s1, __fmul_rn(x[2 * j + 1], x[2 * j + 1]));
            }
            const Sum2 tot = warp_sum(sum_merge(s0, s1), 16);
            const float r = rms_inv(sum_value(tot), (float)kHeadDim, a.eps);
            float qh[8];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                qh[2 * j] = __fmul_rn(__fmul_rn(x[2 * j], r), bf_lo(word(w, j)));
                qh[2 * j + 1] = __fmul_rn(__fmul_rn(x[2 * j + 1], r), bf_hi(word(w, j)));
            }
            float out[8];
            if constexpr (ROPE) {
                const bool first_half = l16 < 8;
                const int base = 8 * (l16 & 7);
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float pe = __shfl_xor_sync(0xffffffffu, qh[e], 8);
                    const float c = cs[base + e], s = sn[base + e];
                    // first half:  q_i c - q_{i+64} s ;  second half: q_{i+64} c + q_i s
                    out[e] = first_half ? __fsub_rn(__fmul_rn(qh[e], c), __fmul_rn(pe, s))
                                        : __fadd_rn(__fmul_rn(qh[e], c), __fmul_rn(pe, s));
                }
            } else {
                const float sc = scale_q;
#pragma unroll
                for (int e = 0; e < 8; ++e)
                    out[e] = isq ? __fmul_rn(qh[e], sc) : qh[e];
            }
            if (act) {
                uint4 o;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    word(o, j) = pack_bf16x2(out[2 * j], out[2 * j + 1]);
                st_global(row + 16 * l16, o);
            }
        }
        __syncthreads();  // cs / sn / scale_q are rewritten for the next token of this CTA
    }
}

// out = bf16(attn * 1/(1 + expf(-(gate + bias_h)))).  One CTA per row, 4 vectors per thread
// per pass, all loads of a pass issued before any arithmetic.
__global__ void __launch_bounds__(256) attn_gate_kernel(const GateArgs a)
{
    const int vpr = (a.n_heads * a.head_dim) >> 3;
    const int vph = a.head_dim >> 3;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
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
                    const float b = a.bias[v / vph];
                    uint4 o;
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float res[2];
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const float g = hh ? bf_hi(word(gv[i], j)) : bf_lo(word(gv[i], j));
                            const float at = hh ? bf_hi(word(av[i], j)) : bf_lo(word(av[i], j));
                            const float z = __fadd_rn(g, b);
                            const float e = expf(-z);
                            const float sig = __fdiv_rn(1.0f, __fadd_rn(1.0f, e));
                            res[hh] = __fmul_rn(at, sig);
                        }
                        word(o, j) = pack_bf16x2(res[0], res[1]);
                    }
                    st_global(out + 16 * (int64_t)v, o);
                }
            }
        }
    }
}

inline unsigned grid_for(int64_t T)
{
    return (unsigned)(T < (int64_t)(1 << 30) ? T : (int64_t)(1 << 30));
}

template <bool ROPE>
cudaError_t launch_qk(const QkArgs &a, cudaStream_t stream)
{
    RopeTable tab;
    for (int i = 0; i < kHalf; ++i)
        tab.inv_freq[i] = ROPE ? a.inv_freq_host[i] : 0.0f;
    const int nheads = a.n_q + a.n_kv;
    int threads = 16 * (nheads < 64 ? nheads : 64);
    threads = (threads + 31) / 32 * 32;
    qk_norm_kernel<ROPE><<<grid_for(a.T), threads, 0, stream>>>(a, tab);
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
