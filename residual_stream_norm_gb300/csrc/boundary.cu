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
// 路由").  Nothing between the stages goes back to HBM: per row the kernel reads x (or the K
// expert rows) and h once, the weights from L1/L2, and writes h' and y once.
//
// Layout: one CTA per token row (grid-stride over rows), each thread owns VPT 16-byte vectors
// of the row at vector indices tid + i * blockDim.x (coalesced).  The row stays in registers as
// packed BF16 between the two block reductions.

#include "beam_device.cuh"
#include "beam_kernels.h"

namespace beam {
namespace {

constexpr int kMaxK = 16;

template <int VPT, bool MOE>
__global__ void __launch_bounds__(VPT >= 4 ? 256 : 1024) boundary_kernel(const BoundaryArgs a)
{
    __shared__ Sum2 red[2][32];
    const int nvec = a.H >> 3;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const float Hf = (float)a.H;
    const uint4 zero = make_uint4(0u, 0u, 0u, 0u);

    for (int64_t row = blockIdx.x; row < a.T; row += gridDim.x) {
        const int64_t row_off = row * (int64_t)a.H;  // elements
        const char *h_in = (const char *)a.h_in + 2 * row_off;
        uint4 xv[VPT], hv[VPT];

        if constexpr (MOE) {
            // c_k = fp32(w_k * routed_scaling); x = bf16(sum_k c_k e_k), one FMA per slot in
            // slot order from +0.
            float c[kMaxK];
#pragma unroll
            for (int k = 0; k < kMaxK; ++k)
                c[k] = k < a.K ? __fmul_rn(a.topk_w[row * a.K + k], a.routed_scaling) : 0.0f;
            const char *e_row = (const char *)a.expert_out + 2 * row_off * a.K;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int v = tid + i * nt;
                if (v < nvec) {
                    hv[i] = ld_stream(h_in + 16 * (int64_t)v);
                    float acc[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j)
                        acc[j] = 0.0f;
#pragma unroll
                    for (int k = 0; k < kMaxK; ++k) {
                        if (k < a.K) {
                            uint4 ev = ld_stream(e_row + 2 * (int64_t)k * a.H + 16 * (int64_t)v);
#pragma unroll
                            for (int j = 0; j < 4; ++j) {
                                acc[2 * j] = __fmaf_rn(c[k], bf_lo(word(ev, j)), acc[2 * j]);
                                acc[2 * j + 1] = __fmaf_rn(c[k], bf_hi(word(ev, j)), acc[2 * j + 1]);
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        word(xv[i], j) = pack_bf16x2(acc[2 * j], acc[2 * j + 1]);
                } else {
                    xv[i] = zero;
                    hv[i] = zero;
                }
            }
        } else {
            const char *x_in = (const char *)a.x_in + 2 * row_off;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int v = tid + i * nt;
                if (v < nvec) {
                    xv[i] = ld_stream(x_in + 16 * (int64_t)v);
                    hv[i] = ld_stream(h_in + 16 * (int64_t)v);
                } else {
                    xv[i] = zero;
                    hv[i] = zero;
                }
            }
        }

        // ---- a1: r = 1/sqrt(mean(x^2) + eps) -----------------------------------------------
        Sum2 s0 = {0.0f, 0.0f}, s1 = {0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float x0 = bf_lo(word(xv[i], j)), x1 = bf_hi(word(xv[i], j));
                sum_add(s0, __fmul_rn(x0, x0));
                sum_add(s1, __fmul_rn(x1, x1));
            }
        }
        const float r = rms_inv(block_sum(sum_merge(s0, s1), red[0]), Hf, a.eps);

        // ---- a1 / a2: xhat = bf16((x r) w_post); h' = bf16(bf16(alpha h) + bf16(xhat / s)) ---
        uint4 hp[VPT];
        s0 = {0.0f, 0.0f};
        s1 = {0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int v = tid + i * nt;
            hp[i] = zero;
            if (v < nvec) {
                const uint4 wv = ld_cached((const char *)a.w_post + 16 * (int64_t)v);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t xw = word(xv[i], j), ww = word(wv, j), hw = word(hv[i], j);
                    const uint32_t xh =
                        pack_bf16x2(__fmul_rn(__fmul_rn(bf_lo(xw), r), bf_lo(ww)),
                                    __fmul_rn(__fmul_rn(bf_hi(xw), r), bf_hi(ww)));
                    const uint32_t bw =
                        pack_bf16x2(__fdiv_rn(bf_lo(xh), a.s), __fdiv_rn(bf_hi(xh), a.s));
                    const uint32_t aw =
                        pack_bf16x2(__fmul_rn(a.alpha, bf_lo(hw)), __fmul_rn(a.alpha, bf_hi(hw)));
                    const uint32_t hq = pack_bf16x2(__fadd_rn(bf_lo(aw), bf_lo(bw)),
                                                    __fadd_rn(bf_hi(aw), bf_hi(bw)));
                    word(hp[i], j) = hq;
                    const float q0 = bf_lo(hq), q1 = bf_hi(hq);
                    sum_add(s0, __fmul_rn(q0, q0));
                    sum_add(s1, __fmul_rn(q1, q1));
                }
            }
        }
        const float r2 = rms_inv(block_sum(sum_merge(s0, s1), red[1]), Hf, a.eps);

        // ---- a3: y = bf16((h' r') w_pre); store h' and y ---------------------------------------
        char *h_out = (char *)a.h_out + 2 * row_off;
        char *y_out = (char *)a.y_out + 2 * row_off;
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int v = tid + i * nt;
            if (v < nvec) {
                const uint4 wv = ld_cached((const char *)a.w_pre + 16 * (int64_t)v);
                uint4 yv;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t hq = word(hp[i], j), ww = word(wv, j);
                    word(yv, j) = pack_bf16x2(__fmul_rn(__fmul_rn(bf_lo(hq), r2), bf_lo(ww)),
                                              __fmul_rn(__fmul_rn(bf_hi(hq), r2), bf_hi(ww)));
                }
                st_global(h_out + 16 * (int64_t)v, hp[i]);
                st_global(y_out + 16 * (int64_t)v, yv);
            }
        }
        if (tid == 0 && a.rstd_out)
            reinterpret_cast<float2 *>(a.rstd_out)[row] = make_float2(r, r2);
        __syncthreads();  // `red` is reused by the next row of this CTA
    }
}

int pick_vpt(int nvec, int max_threads)
{
    int vpt = 1;
    while (vpt < 8 && (nvec + vpt - 1) / vpt > max_threads)
        vpt *= 2;
    return vpt;
}

template <bool MOE>
cudaError_t launch(const BoundaryArgs &a, cudaStream_t stream)
{
    const int nvec = a.H / 8;
    // Few rows: spread each row over many threads (latency); many rows: fewer, fatter threads
    // so several CTAs per SM keep loads in flight.
    const bool small = a.T < 2 * 152;
    const int max_threads = small ? 1024 : (MOE ? 320 : 256);
    const int vpt = pick_vpt(nvec, max_threads);
    int threads = (nvec + vpt - 1) / vpt;
    threads = (threads + 31) / 32 * 32;
    const int64_t grid64 = a.T < (int64_t)(1 << 30) ? a.T : (int64_t)(1 << 30);
    const dim3 grid((unsigned)grid64);
    switch (vpt) {
    case 1: boundary_kernel<1, MOE><<<grid, threads, 0, stream>>>(a); break;
    case 2: boundary_kernel<2, MOE><<<grid, threads, 0, stream>>>(a); break;
    case 4: boundary_kernel<4, MOE><<<grid, threads, 0, stream>>>(a); break;
    default: boundary_kernel<8, MOE><<<grid, threads, 0, stream>>>(a); break;
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_boundary(const BoundaryArgs &a, cudaStream_t stream)
{
    return launch<false>(a, stream);
}

cudaError_t launch_moe_boundary(const BoundaryArgs &a, cudaStream_t stream)
{
    return launch<true>(a, stream);
}

}  // namespace beam
