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
// expert rows) and h once and writes h' and y once; the norm weights come from L1/L2.
//
// Two layouts, same arithmetic (boundary_chain):
//  * rows kernel (few tokens, e.g. batch-1 decode): one CTA per token row; each thread owns VPT
//    16-byte vectors at vector indices tid + i * blockDim.x and loads them straight from memory.
//  * ring kernel (many tokens): a persistent grid (SM count x CTAs per SM) in which each CTA
//    walks its rows through a ring of shared-memory stages.  One thread issues bulk TMA copies
//    (cp.async.bulk, completion on an mbarrier) of the next rows' inputs -- the x row or the K
//    expert rows, and the h row -- so several rows' copies are in flight while the current row
//    is reduced; a stage is refilled as soon as the first block reduction shows that every
//    thread has read it.  Each thread keeps its slice of both norm weights in registers.
// The row stays in registers as packed BF16 between the two block reductions; element math runs
// on packed FP32 pairs (beam_f32x2.cuh) with the same IEEE roundings as the scalar definition.

#include <mutex>

#include "beam_device.cuh"
#include "beam_f32x2.cuh"
#include "beam_kernels.h"
#include "beam_tma.cuh"

namespace beam {

// Fault word of this library on each device; bits are kFault* values (beam_tma.cuh).
__device__ unsigned int g_fault_word = 0u;

namespace {

constexpr int kMaxK = 16;

// Block-wide sum; every warp combines the per-warp partials with the same butterfly, so all
// threads get identical bits.  `slot` holds >= 32 entries not used by a concurrent reduction.
__device__ __forceinline__ float block_sum_w(Sum2 a, Sum2 *slot)
{
    a = warp_sum(a);
    const int lane = threadIdx.x & 31;
    const int nw = blockDim.x >> 5;
    if (lane == 0)
        slot[threadIdx.x >> 5] = a;
    __syncthreads();
    const Sum2 p = lane < nw ? slot[lane] : Sum2{0.0f, 0.0f};
    return sum_value(warp_sum(p));
}

__device__ __forceinline__ Sum2 lanes_merged(const Sum2x2 &a)
{
    return sum_merge(Sum2{lo_of(a.hi), lo_of(a.lo)}, Sum2{hi_of(a.hi), hi_of(a.lo)});
}

// True when every BF16 element of this thread's post-norm weight slice has |w| < 2^120, so
// xhat = bf16((x r) w) cannot overflow and the Markstein division step is safe for it.
template <int VPT>
__device__ __forceinline__ bool weights_small(const uint4 (&w)[VPT])
{
    constexpr uint32_t kCeil = (kWeightMaxExp << 7) | (kWeightMaxExp << 23);
    uint32_t any = 0u;
#pragma unroll
    for (int i = 0; i < VPT; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
            any |= ((word(w[i], j) & 0x7f807f80u) | 0x80008000u) - kCeil;
    return (any & 0x80008000u) == 0u;
}

// The boundary chain for one row whose inputs sit in registers (xv: x, hv: h; wpo / wpr: this
// thread's slices of the weights).  `after_first_sum` runs right after the first block
// reduction (the ring kernel refills its stage there).  `fast_div`: the thread may use the
// Markstein step for x_hat / s (n small enough and its weights small).
template <int VPT, typename AfterFirstSum>
__device__ __forceinline__ void boundary_chain(const BoundaryArgs &a, int64_t row,
                                               const uint4 (&xv)[VPT], const uint4 (&hv)[VPT],
                                               const uint4 (&wpo)[VPT], const uint4 (&wpr)[VPT],
                                               bool fast_div, Sum2 (*red)[32],
                                               AfterFirstSum after_first_sum)
{
    const int nvec = a.H >> 3;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const int64_t row_off = row * (int64_t)a.H;

    // ---- a1: r = 1/sqrt(mean(x^2) + eps) ---------------------------------------------------
    Sum2x2 acc = {0ull, 0ull};
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const f2 x = widen(word(xv[i], j));
            sum2_add(acc, mul2(x, x));
        }
    }
    const float r = rms_inv(block_sum_w(lanes_merged(acc), red[0]), (float)a.H, a.eps);
    after_first_sum();

    // ---- a1 / a2: xhat = bf16((x r) w_post); h' = bf16(bf16(alpha h) + bf16(xhat / s)) -----
    const f2 rr = splat(r), al = splat(a.alpha), ys = splat(a.inv_s), ns = splat(-a.s);
    uint4 hp[VPT];
    acc = {0ull, 0ull};
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int v = tid + i * nt;
        hp[i] = make_uint4(0u, 0u, 0u, 0u);
        if (v < nvec) {
            uint32_t xh[4], bw[4];
            uint32_t floor_all = 0xffffffffu;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                xh[j] = narrow(mul2(mul2(widen(word(xv[i], j)), rr), widen(word(wpo[i], j))));
                exp_floor_check(floor_all, xh[j]);
            }
            if (fast_div && exp_floor_ok(floor_all)) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    bw[j] = narrow(div2_markstein(widen(xh[j]), ns, ys));
            } else {  // zero / tiny / non-finite operands, large n or huge weights
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const f2 q = widen(xh[j]);
                    bw[j] = narrow(make_f2(__fdiv_rn(lo_of(q), a.s), __fdiv_rn(hi_of(q), a.s)));
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint32_t aw = narrow(mul2(al, widen(word(hv[i], j))));
                const uint32_t hq = narrow(add2(widen(aw), widen(bw[j])));
                word(hp[i], j) = hq;
                const f2 hf = widen(hq);
                sum2_add(acc, mul2(hf, hf));
            }
        }
    }
    const f2 rr2 = splat(rms_inv(block_sum_w(lanes_merged(acc), red[1]), (float)a.H, a.eps));

    // ---- a3: y = bf16((h' r') w_pre); store h' and y -----------------------------------------
    char *h_out = (char *)a.h_out + 2 * row_off;
    char *y_out = (char *)a.y_out + 2 * row_off;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int v = tid + i * nt;
        if (v < nvec) {
            uint4 yv;
#pragma unroll
            for (int j = 0; j < 4; ++j)
                word(yv, j) = narrow(mul2(mul2(widen(word(hp[i], j)), rr2), widen(word(wpr[i], j))));
            st_global(h_out + 16 * (int64_t)v, hp[i]);
            st_global(y_out + 16 * (int64_t)v, yv);
        }
    }
    if (tid == 0 && a.rstd_out)
        reinterpret_cast<float2 *>(a.rstd_out)[row] = make_float2(r, lo_of(rr2));
}

// x = bf16(sum_k c_k e_k) for one 16-byte vector: one FMA per slot in slot order from +0.
// `e0` points at slot 0 of this vector; slots are `slot_bytes` apart.
template <bool SMEM>
__device__ __forceinline__ uint4 combine_vec(const float (&c)[kMaxK], int K,
                                             const unsigned char *e0, size_t slot_bytes)
{
    f2 acc[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int k = 0; k < kMaxK; ++k) {
        if (k < K) {
            const unsigned char *p = e0 + (size_t)k * slot_bytes;
            const uint4 ev = SMEM ? *reinterpret_cast<const uint4 *>(p) : ld_stream(p);
            const f2 ck = splat(c[k]);
#pragma unroll
            for (int j = 0; j < 4; ++j)
                acc[j] = fma2(ck, widen(word(ev, j)), acc[j]);
        }
    }
    uint4 x;
#pragma unroll
    for (int j = 0; j < 4; ++j)
        word(x, j) = narrow(acc[j]);
    return x;
}

template <int VPT>
__device__ __forceinline__ void load_weights(const BoundaryArgs &a, uint4 (&wpo)[VPT],
                                             uint4 (&wpr)[VPT])
{
    const int nvec = a.H >> 3;
#pragma unroll
    for (int i = 0; i < VPT; ++i) {
        const int v = threadIdx.x + i * blockDim.x;
        wpo[i] = v < nvec ? ld_cached((const char *)a.w_post + 16 * (int64_t)v) : make_uint4(0u, 0u, 0u, 0u);
        wpr[i] = v < nvec ? ld_cached((const char *)a.w_pre + 16 * (int64_t)v) : make_uint4(0u, 0u, 0u, 0u);
    }
}

// ---- rows kernel: one CTA per row, inputs straight from memory ------------------------------

template <int VPT, bool MOE>
__global__ void __launch_bounds__(VPT == 1 ? 1024 : (VPT == 8 ? 256 : 512))
    boundary_rows_kernel(const BoundaryArgs a)
{
    __shared__ Sum2 red[2][32];
    const int nvec = a.H >> 3;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    uint4 wpo[VPT], wpr[VPT];
    load_weights<VPT>(a, wpo, wpr);
    const bool fast_div = a.fast_div_n && weights_small<VPT>(wpo);

    for (int64_t row = blockIdx.x; row < a.T; row += gridDim.x) {
        const int64_t row_off = row * (int64_t)a.H;
        const char *h_in = (const char *)a.h_in + 2 * row_off;
        uint4 xv[VPT], hv[VPT];
        float c[kMaxK];
        if constexpr (MOE) {
#pragma unroll
            for (int k = 0; k < kMaxK; ++k)
                c[k] = k < a.K ? __fmul_rn(a.topk_w[row * a.K + k], a.routed_scaling) : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int v = tid + i * nt;
            if (v < nvec) {
                hv[i] = ld_stream(h_in + 16 * (int64_t)v);
                if constexpr (MOE)
                    xv[i] = combine_vec<false>(c, a.K, (const unsigned char *)a.expert_out +
                                                           2 * row_off * a.K + 16 * (int64_t)v,
                                               2 * (size_t)a.H);
                else
                    xv[i] = ld_stream((const char *)a.x_in + 2 * row_off + 16 * (int64_t)v);
            } else {
                xv[i] = make_uint4(0u, 0u, 0u, 0u);
                hv[i] = xv[i];
            }
        }
        boundary_chain<VPT>(a, row, xv, hv, wpo, wpr, fast_div, red, [] {});
    }
}

// ---- ring kernel: persistent CTAs, TMA bulk copies through shared-memory stages -------------

constexpr int kRingHeader = 128;  // the stages' mbarriers live in the first 128 bytes

template <int VPT, bool MOE>
__global__ void __launch_bounds__(VPT == 1 ? 1024 : 512)
    boundary_ring_kernel(const BoundaryArgs a, int stages, uint32_t stage_bytes)
{
    extern __shared__ __align__(128) unsigned char dyn[];
    uint64_t *full = reinterpret_cast<uint64_t *>(dyn);
    unsigned char *ring = dyn + kRingHeader;
    __shared__ Sum2 red[2][32];

    const int nvec = a.H >> 3;
    const int tid = threadIdx.x;
    const int nt = blockDim.x;
    const uint32_t row_bytes = 2u * (uint32_t)a.H;
    const int K = MOE ? a.K : 1;
    const uint32_t in_bytes = (uint32_t)K * row_bytes;  // the x row, or the K expert rows
    const int64_t first = blockIdx.x;
    const int64_t stride = gridDim.x;
    const int64_t my_rows = first < a.T ? (a.T - first + stride - 1) / stride : 0;

    auto issue = [&](int64_t i) {  // one thread: fill stage i % stages with row i's inputs
        const int st = (int)(i % stages);
        const int64_t row = first + i * stride;
        unsigned char *dst = ring + (size_t)st * stage_bytes;
        const char *src = MOE ? (const char *)a.expert_out + (size_t)row * in_bytes
                              : (const char *)a.x_in + (size_t)row * row_bytes;
        mbar_arrive_expect_tx(&full[st], in_bytes + row_bytes);
        bulk_g2s(dst, src, in_bytes, &full[st]);
        bulk_g2s(dst + in_bytes, (const char *)a.h_in + (size_t)row * row_bytes, row_bytes,
                 &full[st]);
    };

    if (tid == 0) {
        for (int st = 0; st < stages; ++st)
            mbar_init(&full[st], 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (tid == 0) {
        const int64_t pre = my_rows < stages ? my_rows : stages;
        for (int64_t i = 0; i < pre; ++i)
            issue(i);
    }
    uint4 wpo[VPT], wpr[VPT];
    load_weights<VPT>(a, wpo, wpr);
    const bool fast_div = a.fast_div_n && weights_small<VPT>(wpo);

    float c[kMaxK];
    for (int64_t i = 0; i < my_rows; ++i) {
        const int st = (int)(i % stages);
        const bool ok = mbar_wait(&full[st], (uint32_t)((i / stages) & 1));
        if (__syncthreads_or(!ok)) {
            // Give up: wait (bounded) for this CTA's copies still in flight, flag, return.
            if (tid == 0) {
                const int64_t last = i + stages < my_rows ? i + stages : my_rows;
                for (int64_t j = i; j < last; ++j)
                    (void)mbar_wait(&full[j % stages], (uint32_t)((j / stages) & 1));
                atomicOr(&g_fault_word, kFaultCopyTimeout);
            }
            return;
        }
        const unsigned char *stage = ring + (size_t)st * stage_bytes;
        const int64_t row = first + i * stride;
        if constexpr (MOE) {
#pragma unroll
            for (int k = 0; k < kMaxK; ++k)
                c[k] = k < K ? __fmul_rn(a.topk_w[row * K + k], a.routed_scaling) : 0.0f;
        }
        uint4 xv[VPT], hv[VPT];
#pragma unroll
        for (int j = 0; j < VPT; ++j) {
            const int v = tid + j * nt;
            if (v < nvec) {
                hv[j] = *reinterpret_cast<const uint4 *>(stage + in_bytes + 16 * v);
                if constexpr (MOE)
                    xv[j] = combine_vec<true>(c, K, stage + 16 * v, row_bytes);
                else
                    xv[j] = *reinterpret_cast<const uint4 *>(stage + 16 * v);
            } else {
                xv[j] = make_uint4(0u, 0u, 0u, 0u);
                hv[j] = xv[j];
            }
        }
        // After the first block reduction every thread has read this stage: refill it.
        boundary_chain<VPT>(a, row, xv, hv, wpo, wpr, fast_div, red, [&] {
            if (tid == 0 && i + stages < my_rows)
                issue(i + stages);
        });
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

template <int VPT, bool MOE>
cudaError_t launch_ring(const BoundaryArgs &a, int stages, uint32_t stage_bytes, int threads,
                        int sms, cudaStream_t stream)
{
    const size_t smem = kRingHeader + (size_t)stages * stage_bytes;
    auto kern = boundary_ring_kernel<VPT, MOE>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess)
        return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess)
        return e;
    if (per_sm < 1)
        return cudaErrorInvalidConfiguration;
    const int64_t slots = (int64_t)sms * per_sm;
    const unsigned grid = (unsigned)(a.T < slots ? a.T : slots);
    kern<<<grid, threads, smem, stream>>>(a, stages, stage_bytes);
    return cudaGetLastError();
}

// Smallest vectors-per-thread whose thread count fits both `max_threads` and the kernel's
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

// Below the 227 KB per-block limit, leaving room for static shared memory.
constexpr size_t kMaxDynSmem = 220 * 1024;

template <bool MOE>
cudaError_t launch(const BoundaryArgs &a, cudaStream_t stream)
{
    const int nvec = a.H / 8;
    const int sms = device_sms();
    // Many rows: the persistent TMA ring, when at least two stages of inputs fit in smem.
    if (a.T >= 4 * (int64_t)sms) {
        const uint32_t row_bytes = 2u * (uint32_t)a.H;
        const uint32_t stage_bytes =
            ((MOE ? (uint32_t)a.K + 1u : 2u) * row_bytes + 127u) / 128u * 128u;
        const int max_stages = MOE ? 2 : 4;
        int stages = (int)((kMaxDynSmem - kRingHeader) / stage_bytes);
        stages = stages > max_stages ? max_stages : stages;
        if (stages >= 2) {
            if (MOE && nvec <= 1024)
                return launch_ring<1, MOE>(a, stages, stage_bytes, round_warps(nvec), sms, stream);
            if (nvec <= 1024)
                return launch_ring<2, MOE>(a, stages, stage_bytes, round_warps((nvec + 1) / 2),
                                           sms, stream);
            return launch_ring<4, MOE>(a, stages, stage_bytes, round_warps((nvec + 3) / 4), sms,
                                       stream);
        }
    }
    // Few rows (or inputs too large to stage): one CTA per row straight from memory.
    const bool small = a.T < 2 * (int64_t)sms;
    const int max_threads = small ? 1024 : (MOE ? 320 : 256);
    const int vpt = pick_vpt(nvec, max_threads);
    const int threads = round_warps((nvec + vpt - 1) / vpt);
    const dim3 grid((unsigned)(a.T < (int64_t)(1 << 30) ? a.T : (int64_t)(1 << 30)));
    switch (vpt) {
    case 1: boundary_rows_kernel<1, MOE><<<grid, threads, 0, stream>>>(a); break;
    case 2: boundary_rows_kernel<2, MOE><<<grid, threads, 0, stream>>>(a); break;
    case 4: boundary_rows_kernel<4, MOE><<<grid, threads, 0, stream>>>(a); break;
    default: boundary_rows_kernel<8, MOE><<<grid, threads, 0, stream>>>(a); break;
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
