// beam_api.cu -- C ABI of libbeam_boundary.so: argument checks, host-side coefficients, launch.
//
// Every check runs before any CUDA call, so a rejected call launches nothing, touches no output
// and needs no GPU.  The library holds no state besides small caches (per thread: the RoPE
// frequency table and the residual rule of the last call; per device: the SM count and the
// persistent kernels' launch shapes).  It never allocates device memory, and no call
// synchronises except the beam_device_faults diagnostic.

#include <cmath>
#include <cstdint>
#include <cstring>

#include "../../include/beam_boundary.h"
#include "beam_kernels.h"
#include "beam_exact.cuh"
#include "beam_exp.cuh"
#include "beam_f32x2.cuh"
#include "beam_sincos.cuh"
#include "beam_tma.cuh"

namespace {

constexpr int32_t kMaxHidden = 16384;
constexpr int32_t kMaxK = 16;
constexpr int32_t kHeadDim = 128;
constexpr int32_t kMaxHeads = 1024;

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline int cuda_status(cudaError_t e) { return e == cudaSuccess ? BEAM_OK : BEAM_ERR_CUDA; }

int check_hidden(int32_t H) { return (H < 8 || H > kMaxHidden || H % 8 != 0) ? BEAM_ERR_INVALID_ARG : BEAM_OK; }

bool bad_eps(float eps) { return !(eps >= 0.0f) || !std::isfinite(eps); }

// Arguments of a boundary launch with the persistent kernels' usual copy-wait limit.
beam::BoundaryArgs boundary_args()
{
    beam::BoundaryArgs a{};
    a.wait_ns = beam::kWaitLimitNs;
    return a;
}

// fp32(theta^(-2i/128)) for i < 64, formed in double.  Cached per thread for the last theta.
const float *rope_inv_freq(float theta)
{
    static thread_local float cached_theta = -1.0f;
    static thread_local float table[kHeadDim / 2];
    if (cached_theta != theta) {
        for (int i = 0; i < kHeadDim / 2; ++i)
            table[i] = (float)std::pow((double)theta, -2.0 * (double)i / (double)kHeadDim);
        cached_theta = theta;
    }
    return table;
}

// The residual operand rule of the boundary kernels for this n (beam_f32x2.cuh).  The check of
// the 128 significands is cached per thread for the last residual index.
void set_residual_rule(beam::BoundaryArgs &a)
{
    static thread_local float cached_s = -1.0f;
    static thread_local bool cached_ok = false;
    a.inv_s = 1.0f / a.s;
    if (a.s != cached_s) {
        cached_ok = beam::residual_mul_exact(a.s, a.inv_s);
        cached_s = a.s;
    }
    a.mul_div = cached_ok;
    const uint32_t f = beam::residual_floor_exp(a.s);
    a.floor_bits = (f << 7) | (f << 23);
}

int check_qk(void *q, void *k, int64_t q_row_stride, int64_t k_row_stride, const void *wq,
             const void *wk, const int64_t *pos, int64_t T, int32_t n_q, int32_t n_kv,
             int32_t head_dim, float eps)
{
    if (head_dim != kHeadDim)
        return BEAM_ERR_UNSUPPORTED;
    if (T < 0 || n_q < 0 || n_kv < 0 || n_q + n_kv < 1 || n_q + n_kv > kMaxHeads || bad_eps(eps))
        return BEAM_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_OK;
    if (!pos || (n_q > 0 && (!q || !wq)) || (n_kv > 0 && (!k || !wk)))
        return BEAM_ERR_INVALID_ARG;
    if ((n_q > 0 && q_row_stride < (int64_t)n_q * kHeadDim) ||
        (n_kv > 0 && k_row_stride < (int64_t)n_kv * kHeadDim))
        return BEAM_ERR_INVALID_ARG;
    if ((n_q > 0 && (!aligned(q, 16) || !aligned(wq, 16) || q_row_stride % 8 != 0)) ||
        (n_kv > 0 && (!aligned(k, 16) || !aligned(wk, 16) || k_row_stride % 8 != 0)) ||
        !aligned(pos, 8))
        return BEAM_ERR_MISALIGNED;
    return BEAM_OK;
}

// The KV-cache arguments of the *_kv_fwd calls; on success fills the cache fields of `a`.
int check_kv(beam::QkArgs &a, const void *v, int64_t v_row_stride, const int64_t *slot_mapping,
             void *k_cache, void *v_cache, int64_t num_slots, int32_t cache_dtype, float k_scale,
             float v_scale, int32_t n_kv)
{
    if (cache_dtype != 0 && cache_dtype != 1)
        return BEAM_ERR_UNSUPPORTED;
    if (num_slots < 0 || (cache_dtype == 1 && (!(k_scale > 0.0f) || !std::isfinite(k_scale) ||
                                               !(v_scale > 0.0f) || !std::isfinite(v_scale))))
        return BEAM_ERR_INVALID_ARG;
    if (n_kv > 0 && (!v || !slot_mapping || !k_cache || !v_cache ||
                     v_row_stride < (int64_t)n_kv * kHeadDim))
        return BEAM_ERR_INVALID_ARG;
    const uintptr_t cache_align = cache_dtype == 0 ? 16 : 8;
    if (n_kv > 0 && (!aligned(v, 16) || v_row_stride % 8 != 0 || !aligned(slot_mapping, 8) ||
                     !aligned(k_cache, cache_align) || !aligned(v_cache, cache_align)))
        return BEAM_ERR_MISALIGNED;
    a.v = v;
    a.v_stride = v_row_stride;
    a.slot = slot_mapping;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.num_slots = num_slots;
    a.cache_mode = n_kv > 0 ? 1 + cache_dtype : 0;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    int ek, ev;
    a.k_pow2 = std::frexp(k_scale, &ek) == 0.5f;
    a.v_pow2 = std::frexp(v_scale, &ev) == 0.5f;
    a.k_inv = a.k_pow2 ? std::ldexp(1.0f, 1 - ek) : 0.0f;
    a.v_inv = a.v_pow2 ? std::ldexp(1.0f, 1 - ev) : 0.0f;
    return BEAM_OK;
}

}  // namespace

extern "C" {

int beam_abi_version(void) { return BEAM_ABI_VERSION; }

const char *beam_status_str(int status)
{
    switch (status) {
    case BEAM_OK: return "BEAM_OK";
    case BEAM_ERR_INVALID_ARG: return "BEAM_ERR_INVALID_ARG";
    case BEAM_ERR_MISALIGNED: return "BEAM_ERR_MISALIGNED";
    case BEAM_ERR_UNSUPPORTED: return "BEAM_ERR_UNSUPPORTED";
    case BEAM_ERR_CUDA: return "BEAM_ERR_CUDA";
    default: return "unknown";
    }
}

int beam_residual_scales(int32_t n, float *alpha, float *s)
{
    if (n < 1 || !alpha || !s)
        return BEAM_ERR_INVALID_ARG;
    *alpha = (float)std::sqrt((double)(n - 1) / (double)n);
    *s = (float)std::sqrt((double)n);
    return BEAM_OK;
}

int beam_device_faults(uint32_t *flags, int clear)
{
    if (!flags)
        return BEAM_ERR_INVALID_ARG;
    unsigned int v = 0u;
    const cudaError_t e = beam::read_fault_word(&v, clear != 0);
    *flags = v;
    return cuda_status(e);
}

int beam_selftest_copy_timeout(int64_t limit_ns, cudaStream_t stream)
{
    if (limit_ns < 1000 || limit_ns > 2000000000)
        return BEAM_ERR_INVALID_ARG;
    return cuda_status(beam::launch_copy_timeout_selftest((unsigned long long)limit_ns, stream));
}

int beam_residual_operand(const float *x, float *b_out, int64_t count, int32_t n)
{
    if (n < 1 || count < 0 || (count > 0 && (!x || !b_out)))
        return BEAM_ERR_INVALID_ARG;
    beam::BoundaryArgs a{};
    beam_residual_scales(n, &a.alpha, &a.s);
    set_residual_rule(a);
    const uint32_t f = a.floor_bits >> 23;
    int st = BEAM_OK;
    for (int64_t i = 0; i < count; ++i) {
        uint32_t u;
        std::memcpy(&u, &x[i], sizeof u);
        if (u & 0xffffu) {  // not a BF16 value
            b_out[i] = NAN;
            st = BEAM_ERR_INVALID_ARG;
            continue;
        }
        b_out[i] = beam::residual_operand_host(x[i], a.s, a.inv_s, a.mul_div, f);
    }
    return st;
}

int beam_exact_square_sum(const float *v, int64_t count, float *out)
{
    if (count < 0 || count > 16384 || !out || (count > 0 && !v))
        return BEAM_ERR_INVALID_ARG;
    uint32_t mx = 0;  // bits of the largest square (NaN above +inf)
    for (int64_t i = 0; i < count; ++i) {
        const float sq = v[i] * v[i];
        uint32_t u;
        std::memcpy(&u, &sq, sizeof u);
        u &= 0x7fffffffu;
        mx = u > mx ? u : mx;
    }
    if (mx >= 0x7f800000u) {
        *out = mx > 0x7f800000u ? NAN : INFINITY;
        return BEAM_OK;
    }
    if (mx == 0) {
        *out = 0.0f;
        return BEAM_OK;
    }
    const uint32_t emax = beam::exact_emax(mx);
    beam::ExactAcc a{0, 0, 0};
    for (int64_t i = 0; i < count; ++i) {
        const float sq = v[i] * v[i];
        uint32_t u;
        std::memcpy(&u, &sq, sizeof u);
        beam::exact_add(a, u, emax);
    }
    *out = beam::exact_round(a, emax);
    return BEAM_OK;
}

int beam_routing_sigmoid(const float *z, float *out, int64_t count)
{
    if (count < 0 || (count > 0 && (!z || !out)))
        return BEAM_ERR_INVALID_ARG;
    for (int64_t i = 0; i < count; ++i)
        out[i] = beam::sigmoid_rounded(z[i]);
    return BEAM_OK;
}

int beam_rope_cos_sin(const float *angle, float *cos_out, float *sin_out, int64_t count)
{
    if (count < 0 || (count > 0 && (!angle || !cos_out || !sin_out)))
        return BEAM_ERR_INVALID_ARG;
    int st = BEAM_OK;
    for (int64_t i = 0; i < count; ++i) {
        const float x = angle[i];
        if (!(std::fabs(x) < beam::kSinCosMaxArg)) {
            cos_out[i] = sin_out[i] = NAN;
            st = BEAM_ERR_INVALID_ARG;
            continue;
        }
        beam::sincos_rounded(x, &sin_out[i], &cos_out[i]);
    }
    return st;
}

int beam_boundary_fwd(void *h_out, void *y_out, const void *h_in, const void *x_in,
                      const void *w_post, const void *w_pre, int64_t T, int32_t H, int32_t n,
                      float eps, float *rstd_out, cudaStream_t stream)
{
    if (T < 0 || n < 1 || bad_eps(eps) || check_hidden(H) != BEAM_OK)
        return BEAM_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_OK;
    if (!h_out || !y_out || !h_in || !x_in || !w_post || !w_pre)
        return BEAM_ERR_INVALID_ARG;
    if (!aligned(h_out, 16) || !aligned(y_out, 16) || !aligned(h_in, 16) || !aligned(x_in, 16) ||
        !aligned(w_post, 16) || !aligned(w_pre, 16) || (rstd_out && !aligned(rstd_out, 8)))
        return BEAM_ERR_MISALIGNED;
    beam::BoundaryArgs a = boundary_args();
    a.h_out = h_out;
    a.y_out = y_out;
    a.h_in = h_in;
    a.x_in = x_in;
    a.w_post = w_post;
    a.w_pre = w_pre;
    a.rstd_out = rstd_out;
    a.T = T;
    a.H = H;
    a.K = 0;
    a.eps = eps;
    beam_residual_scales(n, &a.alpha, &a.s);
    set_residual_rule(a);
    return cuda_status(beam::launch_boundary(a, stream));
}

int beam_moe_combine_boundary_fwd(void *h_out, void *y_out, const void *h_in,
                                  const void *expert_out, const float *topk_w,
                                  float routed_scaling, const void *w_post, const void *w_pre,
                                  int64_t T, int32_t H, int32_t K, int32_t n, float eps,
                                  float *rstd_out, cudaStream_t stream)
{
    if (T < 0 || n < 1 || K < 1 || K > kMaxK || bad_eps(eps) || !std::isfinite(routed_scaling) ||
        check_hidden(H) != BEAM_OK)
        return BEAM_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_OK;
    if (!h_out || !y_out || !h_in || !expert_out || !topk_w || !w_post || !w_pre)
        return BEAM_ERR_INVALID_ARG;
    if (!aligned(h_out, 16) || !aligned(y_out, 16) || !aligned(h_in, 16) ||
        !aligned(expert_out, 16) || !aligned(topk_w, 4) || !aligned(w_post, 16) ||
        !aligned(w_pre, 16) || (rstd_out && !aligned(rstd_out, 8)))
        return BEAM_ERR_MISALIGNED;
    beam::BoundaryArgs a = boundary_args();
    a.h_out = h_out;
    a.y_out = y_out;
    a.h_in = h_in;
    a.expert_out = expert_out;
    a.topk_w = topk_w;
    a.routed_scaling = routed_scaling;
    a.w_post = w_post;
    a.w_pre = w_pre;
    a.rstd_out = rstd_out;
    a.T = T;
    a.H = H;
    a.K = K;
    a.eps = eps;
    beam_residual_scales(n, &a.alpha, &a.s);
    set_residual_rule(a);
    return cuda_status(beam::launch_moe_boundary(a, stream));
}

int beam_allreduce_boundary_fwd(void *h_out, void *y_out, const void *h_in,
                                const void *const *x_parts, int32_t P, const void *w_post,
                                const void *w_pre, int64_t T, int32_t H, int32_t n, float eps,
                                float *rstd_out, cudaStream_t stream)
{
    if (T < 0 || n < 1 || P < 1 || P > beam::kMaxParts || bad_eps(eps) ||
        check_hidden(H) != BEAM_OK)
        return BEAM_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_OK;
    if (!h_out || !y_out || !h_in || !x_parts || !w_post || !w_pre)
        return BEAM_ERR_INVALID_ARG;
    for (int32_t p = 0; p < P; ++p)
        if (!x_parts[p])
            return BEAM_ERR_INVALID_ARG;
    if (!aligned(h_out, 16) || !aligned(y_out, 16) || !aligned(h_in, 16) ||
        !aligned(w_post, 16) || !aligned(w_pre, 16) || (rstd_out && !aligned(rstd_out, 8)))
        return BEAM_ERR_MISALIGNED;
    for (int32_t p = 0; p < P; ++p)
        if (!aligned(x_parts[p], 16))
            return BEAM_ERR_MISALIGNED;
    beam::BoundaryArgs a = boundary_args();
    beam::TpParts parts{};
    a.h_out = h_out;
    a.y_out = y_out;
    a.h_in = h_in;
    for (int32_t p = 0; p < P; ++p)
        parts.p[p] = x_parts[p];
    a.P = P;
    a.w_post = w_post;
    a.w_pre = w_pre;
    a.rstd_out = rstd_out;
    a.T = T;
    a.H = H;
    a.eps = eps;
    beam_residual_scales(n, &a.alpha, &a.s);
    set_residual_rule(a);
    return cuda_status(beam::launch_allreduce_boundary(a, parts, stream));
}

int beam_selftest_persistent_timeout(int32_t kind, void *h_out, void *y_out, float *rstd_out,
                                     const void *w_post, const void *w_pre, int64_t T, int32_t H,
                                     int64_t limit_ns, cudaStream_t stream)
{
    if ((kind != 0 && kind != 1) || T < 1 || T > (int64_t)1 << 20 || limit_ns < 1000 ||
        limit_ns > 2000000000 || check_hidden(H) != BEAM_OK || H > 8192)
        return BEAM_ERR_INVALID_ARG;
    if (!h_out || !y_out || !w_post || !w_pre)
        return BEAM_ERR_INVALID_ARG;
    if (!aligned(h_out, 16) || !aligned(y_out, 16) || !aligned(w_post, 16) ||
        !aligned(w_pre, 16) || (rstd_out && !aligned(rstd_out, 8)))
        return BEAM_ERR_MISALIGNED;
    beam::BoundaryArgs a = boundary_args();
    a.h_out = h_out;
    a.y_out = y_out;
    a.w_post = w_post;
    a.w_pre = w_pre;
    a.rstd_out = rstd_out;
    a.T = T;
    a.H = H;
    a.K = kind == 1 ? 8 : 0;
    a.routed_scaling = 1.0f;
    a.eps = 1e-6f;
    a.wait_ns = (unsigned long long)limit_ns;
    beam_residual_scales(2, &a.alpha, &a.s);
    set_residual_rule(a);
    return cuda_status(beam::launch_persistent_starved(a, kind == 1, stream));
}

int beam_qk_norm_rope_fwd(void *q, void *k, int64_t q_row_stride, int64_t k_row_stride,
                          const void *wq, const void *wk, const int64_t *pos, int64_t T,
                          int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, float eps,
                          float theta, cudaStream_t stream)
{
    int st = check_qk(q, k, q_row_stride, k_row_stride, wq, wk, pos, T, n_q_heads, n_kv_heads,
                      head_dim, eps);
    if (st != BEAM_OK)
        return st;
    if (!(theta > 0.0f) || !std::isfinite(theta))
        return BEAM_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_OK;
    beam::QkArgs a{};
    a.q = q;
    a.k = k;
    a.q_stride = q_row_stride;
    a.k_stride = k_row_stride;
    a.wq = wq;
    a.wk = wk;
    a.pos = pos;
    a.T = T;
    a.n_q = n_q_heads;
    a.n_kv = n_kv_heads;
    a.eps = eps;
    a.inv_freq_host = rope_inv_freq(theta);
    return cuda_status(beam::launch_qk_norm_rope(a, stream));
}

int beam_qk_norm_ssmax_fwd(void *q, void *k, int64_t q_row_stride, int64_t k_row_stride,
                           const void *wq, const void *wk, const int64_t *pos, int64_t T,
                           int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, float eps,
                           float ssmax_base, float ssmax_exp, cudaStream_t stream)
{
    int st = check_qk(q, k, q_row_stride, k_row_stride, wq, wk, pos, T, n_q_heads, n_kv_heads,
                      head_dim, eps);
    if (st != BEAM_OK)
        return st;
    if (!(ssmax_base > 0.0f) || !std::isfinite(ssmax_base) || !std::isfinite(ssmax_exp))
        return BEAM_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_OK;
    beam::QkArgs a{};
    a.q = q;
    a.k = k;
    a.q_stride = q_row_stride;
    a.k_stride = k_row_stride;
    a.wq = wq;
    a.wk = wk;
    a.pos = pos;
    a.T = T;
    a.n_q = n_q_heads;
    a.n_kv = n_kv_heads;
    a.eps = eps;
    a.ssmax_base = ssmax_base;
    a.ssmax_exp = ssmax_exp;
    return cuda_status(beam::launch_qk_norm_ssmax(a, stream));
}

int beam_qk_norm_rope_kv_fwd(void *q, void *k, int64_t q_row_stride, int64_t k_row_stride,
                             const void *v, int64_t v_row_stride, const void *wq, const void *wk,
                             const int64_t *pos, const int64_t *slot_mapping, void *k_cache,
                             void *v_cache, int64_t num_slots, int32_t cache_dtype, float k_scale,
                             float v_scale, int64_t T, int32_t n_q_heads, int32_t n_kv_heads,
                             int32_t head_dim, float eps, float theta, cudaStream_t stream)
{
    int st = check_qk(q, k, q_row_stride, k_row_stride, wq, wk, pos, T, n_q_heads, n_kv_heads,
                      head_dim, eps);
    if (st != BEAM_OK)
        return st;
    if (!(theta > 0.0f) || !std::isfinite(theta))
        return BEAM_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_OK;
    beam::QkArgs a{};
    st = check_kv(a, v, v_row_stride, slot_mapping, k_cache, v_cache, num_slots, cache_dtype,
                  k_scale, v_scale, n_kv_heads);
    if (st != BEAM_OK)
        return st;
    a.q = q;
    a.k = k;
    a.q_stride = q_row_stride;
    a.k_stride = k_row_stride;
    a.wq = wq;
    a.wk = wk;
    a.pos = pos;
    a.T = T;
    a.n_q = n_q_heads;
    a.n_kv = n_kv_heads;
    a.eps = eps;
    a.inv_freq_host = rope_inv_freq(theta);
    return cuda_status(beam::launch_qk_norm_rope(a, stream));
}

int beam_qk_norm_ssmax_kv_fwd(void *q, void *k, int64_t q_row_stride, int64_t k_row_stride,
                              const void *v, int64_t v_row_stride, const void *wq, const void *wk,
                              const int64_t *pos, const int64_t *slot_mapping, void *k_cache,
                              void *v_cache, int64_t num_slots, int32_t cache_dtype, float k_scale,
                              float v_scale, int64_t T, int32_t n_q_heads, int32_t n_kv_heads,
                              int32_t head_dim, float eps, float ssmax_base, float ssmax_exp,
                              cudaStream_t stream)
{
    int st = check_qk(q, k, q_row_stride, k_row_stride, wq, wk, pos, T, n_q_heads, n_kv_heads,
                      head_dim, eps);
    if (st != BEAM_OK)
        return st;
    if (!(ssmax_base > 0.0f) || !std::isfinite(ssmax_base) || !std::isfinite(ssmax_exp))
        return BEAM_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_OK;
    beam::QkArgs a{};
    st = check_kv(a, v, v_row_stride, slot_mapping, k_cache, v_cache, num_slots, cache_dtype,
                  k_scale, v_scale, n_kv_heads);
    if (st != BEAM_OK)
        return st;
    a.q = q;
    a.k = k;
    a.q_stride = q_row_stride;
    a.k_stride = k_row_stride;
    a.wq = wq;
    a.wk = wk;
    a.pos = pos;
    a.T = T;
    a.n_q = n_q_heads;
    a.n_kv = n_kv_heads;
    a.eps = eps;
    a.ssmax_base = ssmax_base;
    a.ssmax_exp = ssmax_exp;
    return cuda_status(beam::launch_qk_norm_ssmax(a, stream));
}

int beam_grouped_topk_fwd(int32_t *topk_ids, float *topk_w, const float *logits,
                          const float *bias, int64_t T, int32_t n_experts, int32_t n_groups,
                          int32_t topk_groups, int32_t top_k, cudaStream_t stream)
{
    if (n_experts != 256 || n_groups != 8 || topk_groups != 4 || top_k != 8)
        return BEAM_ERR_UNSUPPORTED;
    if (T < 0)
        return BEAM_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_OK;
    if (!topk_ids || !topk_w || !logits || !bias)
        return BEAM_ERR_INVALID_ARG;
    if (!aligned(logits, 16) || !aligned(bias, 16) || !aligned(topk_ids, 4) ||
        !aligned(topk_w, 4))
        return BEAM_ERR_MISALIGNED;
    beam::RouteArgs a{};
    a.logits = logits;
    a.bias = bias;
    a.ids = topk_ids;
    a.weights = topk_w;
    a.T = T;
    return cuda_status(beam::launch_grouped_topk(a, stream));
}

int beam_attn_gate_fwd(void *out, const void *attn, const void *gate, const float *bias,
                       int64_t T, int32_t n_heads, int32_t head_dim, int64_t attn_row_stride,
                       int64_t gate_row_stride, int64_t out_row_stride, cudaStream_t stream)
{
    if (head_dim < 8 || head_dim > 1024 || head_dim % 8 != 0)
        return BEAM_ERR_UNSUPPORTED;
    if (T < 0 || n_heads < 1 || n_heads > kMaxHeads)
        return BEAM_ERR_INVALID_ARG;
    if (T == 0)
        return BEAM_OK;
    const int64_t C = (int64_t)n_heads * head_dim;
    if (!out || !attn || !gate || !bias || attn_row_stride < C || gate_row_stride < C ||
        out_row_stride < C)
        return BEAM_ERR_INVALID_ARG;
    if (!aligned(out, 16) || !aligned(attn, 16) || !aligned(gate, 16) || !aligned(bias, 4) ||
        attn_row_stride % 8 != 0 || gate_row_stride % 8 != 0 || out_row_stride % 8 != 0)
        return BEAM_ERR_MISALIGNED;
    beam::GateArgs a{};
    a.out = out;
    a.attn = attn;
    a.gate = gate;
    a.bias = bias;
    a.T = T;
    a.n_heads = n_heads;
    a.head_dim = head_dim;
    a.attn_stride = attn_row_stride;
    a.gate_stride = gate_row_stride;
    a.out_stride = out_row_stride;
    a.head_magic = beam::gate_head_magic(head_dim);
    return cuda_status(beam::launch_attn_gate(a, stream));
}

}  // extern "C"
