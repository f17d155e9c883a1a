// beam_kernels.h -- internal launch interface between the C ABI (beam_api.cu) and the kernels.
// Arguments arrive here already validated; launchers only pick a configuration and launch.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace beam {

// Launch with programmatic stream serialisation (see pdl_wait in beam_device.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Largest number of tensor-parallel partials the all-reduce boundary takes.
constexpr int kMaxParts = 16;

struct BoundaryArgs {
    void *h_out;
    void *y_out;
    const void *h_in;
    const void *x_in;        // boundary: sublayer output [T, H]
    const void *expert_out;  // MoE: [T, K, H] (x_in unused)
    const float *topk_w;     // MoE: [T, K]
    const void *w_post;
    const void *w_pre;
    float *rstd_out;         // [T, 2] or nullptr
    int64_t T;
    int32_t H;
    int32_t K;               // 0 for the plain boundary
    int32_t P;               // tensor-parallel partials (0 unless the all-reduce boundary)
    float routed_scaling;
    float alpha;             // fp32(sqrt((n-1)/n))
    float s;                 // fp32(sqrt(n))
    float inv_s;             // y = fp32(1 / s), IEEE division on the host
    bool mul_div;            // residual_mul_exact(s, y): b = bf16(x y) where x is above the floor
    uint32_t floor_bits;     // (f << 7) | (f << 23), f = residual_floor_exp(s)
    float eps;
    unsigned long long wait_ns;  // limit of a persistent kernel's wait on its own copies
};

// The tensor-parallel partials of the all-reduce boundary, a kernel parameter of its own so
// that the other boundary kernels' parameters stay small (they are copied at every launch).
struct TpParts {
    const void *p[kMaxParts];  // P partial sublayer outputs [T, H] each
};

struct QkArgs {
    void *q;
    void *k;
    int64_t q_stride;  // elements
    int64_t k_stride;
    const void *wq;
    const void *wk;
    const int64_t *pos;
    int64_t T;
    int32_t n_q;
    int32_t n_kv;
    float eps;
    // RoPE
    const float *inv_freq_host;  // [64], host memory, copied into the launch parameters
    // SSMax
    float ssmax_base;
    float ssmax_exp;
    // KV-cache write (cache_mode 0: none, 1: BF16, 2: FP8 E4M3 of value / scale)
    const void *v;          // [T, n_kv, 128] rows, v_stride elements apart
    int64_t v_stride;
    const int64_t *slot;    // [T] physical slot per token; < 0 or >= num_slots: not written
    void *k_cache;          // [num_slots, n_kv, 128]
    void *v_cache;
    int64_t num_slots;
    int32_t cache_mode;
    float k_scale, v_scale;
    float k_inv, v_inv;     // 1 / scale, used only where the scale is a power of two
    bool k_pow2, v_pow2;
};

struct RouteArgs {
    const float *logits;  // [T, 256] FP32 router logits
    const float *bias;    // [256] FP32 correction bias
    int32_t *ids;         // [T, 8] chosen experts, best first
    float *weights;       // [T, 8] renormalised sigmoid scores
    int64_t T;
};

struct GateArgs {
    void *out;
    const void *attn;
    const void *gate;
    const float *bias;
    int64_t T;
    int32_t n_heads;
    int32_t head_dim;
    int64_t attn_stride;
    int64_t gate_stride;
    int64_t out_stride;
    uint64_t head_magic;  // gate_head_magic(head_dim)
};

cudaError_t launch_boundary(const BoundaryArgs &a, cudaStream_t stream);
cudaError_t launch_moe_boundary(const BoundaryArgs &a, cudaStream_t stream);
cudaError_t launch_allreduce_boundary(const BoundaryArgs &a, const TpParts &parts,
                                      cudaStream_t stream);
// Runs a persistent boundary kernel (moe: the MoE ring with K slots, else the plain boundary's
// prefetch kernel) with its bulk copies withheld: its first wait runs out after a.wait_ns, it
// raises the fault word and writes nothing.  a.K is the MoE slot count; inputs are not read.
cudaError_t launch_persistent_starved(const BoundaryArgs &a, bool moe, cudaStream_t stream);
cudaError_t launch_qk_norm_rope(const QkArgs &a, cudaStream_t stream);
cudaError_t launch_qk_norm_ssmax(const QkArgs &a, cudaStream_t stream);
cudaError_t launch_attn_gate(const GateArgs &a, cudaStream_t stream);
cudaError_t launch_grouped_topk(const RouteArgs &a, cudaStream_t stream);
// ceil(2^32 / (head_dim / 8)): the multiplier that maps a gate vector index to its head.
uint64_t gate_head_magic(int32_t head_dim);

// Runs the copy-timeout path once: a wait that nothing completes gives up after limit_ns and
// raises bit 0 of the fault word.
cudaError_t launch_copy_timeout_selftest(unsigned long long limit_ns, cudaStream_t stream);

// The device fault word of the current device (bit 0: a kernel gave up waiting for its own bulk
// copies); synchronous.
cudaError_t read_fault_word(unsigned int *value, bool clear);

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace beam
