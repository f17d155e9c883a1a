/*
 * beam_boundary.h -- C ABI of the Beam sublayer-boundary library (libbeam_boundary.so, sm_103a).
 *
 * The library computes the per-token fused path at the sublayer boundaries of the Beam-1.0
 * 501B-A23B MoE decoder, and the two attention-side kernels that sit on the same path.
 *
 * Pages cited (titles as printed):
 *   [vLLM]  "Serving Reflection Beam auf vLLM ab Tag 0"
 *   [SGL]   "SGLang 支撑编程模型 Beam 生产部署"
 *
 * Conventions shared by every call
 * --------------------------------
 *  - BF16 tensors are passed as `void*` to IEEE bfloat16 storage; FP32 tensors as `float*`.
 *  - Every pointer is a device pointer on the CURRENT CUDA device.  The caller allocates, owns
 *    and frees every buffer; the library never allocates or frees memory, and no call
 *    synchronises except the beam_device_faults diagnostic.
 *  - Every call is asynchronous on `stream` (0 = the legacy default stream).  The returned status
 *    reflects the argument checks and `cudaGetLastError()` right after the launch; a fault that
 *    happens later surfaces on the next synchronising CUDA call, as for any kernel.
 *  - Arguments are validated before anything is launched; on any error nothing is launched and
 *    no output is touched.  T == 0 returns BEAM_OK without launching (pointers may then be NULL).
 *  - Alignment: every BF16 pointer 16-byte aligned, row strides multiples of 8 elements (16 B),
 *    `float*` / `int64_t*` arrays aligned to their element size (the per-token FP32 pair
 *    `rstd_out` to 8 bytes).  Violations return BEAM_ERR_MISALIGNED.
 *  - Arithmetic is FP32 with IEEE division and square root; results are rounded to BF16 with
 *    round-to-nearest-even exactly at the points each call lists.
 *  - Aliasing: only the overlaps each call names are allowed; any other overlap is undefined.
 *  - Launch order: kernels are launched with programmatic dependent launch.  A kernel may start
 *    while the preceding kernel on the same stream is still running, and it reads its model
 *    parameters (norm weights w_post / w_pre / wq / wk, the gate bias) before waiting for that
 *    kernel; every other input is read, and every output written, only after the preceding
 *    kernel has completed.  So the norm weights and the gate bias must not be written by the
 *    kernel launched immediately before on the same stream.
 */
#ifndef BEAM_BOUNDARY_H
#define BEAM_BOUNDARY_H

#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define BEAM_ABI_VERSION 2

/* Symbols of this header are the library's only exported symbols. */
#if defined(__GNUC__)
#define BEAM_API __attribute__((visibility("default")))
#else
#define BEAM_API
#endif

typedef enum {
    BEAM_OK = 0,
    BEAM_ERR_INVALID_ARG = -1,  /* NULL pointer, negative size, out-of-range parameter        */
    BEAM_ERR_MISALIGNED = -2,   /* pointer or stride not aligned as the conventions require     */
    BEAM_ERR_UNSUPPORTED = -3,  /* a shape the kernels do not implement (e.g. head_dim != 128)  */
    BEAM_ERR_CUDA = -4          /* the launch failed; see cudaGetLastError() semantics above    */
} beam_status_t;

/* BEAM_ABI_VERSION of the loaded library. */
BEAM_API int beam_abi_version(void);

/* Static, NUL-terminated name of a status code ("BEAM_OK", ...; "unknown" otherwise). */
BEAM_API const char *beam_status_str(int status);

/* Host-only helper: the FP32 coefficients the boundary calls use for residual index n >= 1,
 * alpha = fp32(sqrt((n-1)/n)) and s = fp32(sqrt(n)), each computed in double and rounded once.
 * [vLLM] "MoE und Residual-Stream", bullet "Tiefenskalierte Residuen".
 * Returns BEAM_ERR_INVALID_ARG for n < 1 or NULL outputs. */
BEAM_API int beam_residual_scales(int32_t n, float *alpha, float *s);

/* Fault word of the current device.  The persistent boundary kernels (the many-row plain, MoE
 * and all-reduce boundaries) wait on their own bulk copies with a time limit (2 s).  A CTA whose
 * wait runs out stops issuing copies, writes nothing from then on (rows it had finished before
 * keep their new h', y and rstd; the rest keep their previous contents -- an in-place h stays the
 * old residual stream there), waits (bounded) for its copies still in flight, and sets bit 0
 * (1 = copy wait timed out).  The call itself has already returned BEAM_OK by then: this word is
 * the only signal.  Never set in normal operation.
 * Synchronous (a device-to-host copy on the legacy default stream); `clear` != 0 resets the word.
 * No counterpart on the pages: a diagnostic of this library. */
BEAM_API int beam_device_faults(uint32_t *flags, int clear);

/* Diagnostic: exercises the copy-timeout path of the persistent kernels without a fault.  One
 * CTA arms an mbarrier for 16 bytes that no copy delivers, waits with the kernels' bounded wait
 * for limit_ns nanoseconds (1 us .. 2 s), gives up and sets bit 0 of the device fault word, as a
 * persistent kernel whose copies stalled would; nothing is left in flight.  Asynchronous on `stream`;
 * read the result with beam_device_faults().  BEAM_ERR_INVALID_ARG for a limit out of range. */
BEAM_API int beam_selftest_copy_timeout(int64_t limit_ns, cudaStream_t stream);

/* Diagnostic: runs a persistent boundary kernel -- kind 0: the plain boundary's prefetch kernel;
 * kind 1: the MoE ring with 8 slots -- with its bulk copies withheld (its barriers are armed, no
 * copy is issued), so that its waits run out after limit_ns nanoseconds (1 us .. 2 s) exactly as
 * they would if the copies stalled.  The kernel must then write nothing to h_out, y_out
 * [T, H] and rstd_out [T, 2] (nullable), and set bit 0 of the device fault word.  The norm
 * weights w_post, w_pre [H] are read; no other input is.  T in [1, 2^20], H a multiple of 8 in
 * [8, 8192].  Asynchronous on `stream`.  No counterpart on the pages: a diagnostic of the
 * persistent kernels' time limit. */
BEAM_API int beam_selftest_persistent_timeout(int32_t kind, void *h_out, void *y_out,
                                              float *rstd_out, const void *w_post,
                                              const void *w_pre, int64_t T, int32_t H,
                                              int64_t limit_ns, cudaStream_t stream);

/* Host-only helper: the residual operand b = bf16(x / s), s = fp32(sqrt(n)), returned as FP32
 * values, for `count` BF16 values x given as FP32 (low 16 bits zero) in host memory, exactly as
 * the boundary kernels form it ("Tiefenskalierte Residuen").  The kernels take b = bf16(RN(x y))
 * with y = RN(1/s) when that is known to equal bf16(RN(x / s)) -- for this n, checked over all
 * 128 BF16 significands, and x above an exponent floor so that both values are normal -- and IEEE
 * division otherwise; the result equals bf16 of the IEEE quotient for every BF16 x (checked
 * exhaustively by the tests).  Returns BEAM_ERR_INVALID_ARG for n < 1, count < 0 or NULL
 * arrays, and for inputs that are not BF16 values (their outputs are NaN). */
BEAM_API int beam_residual_operand(const float *x, float *b_out, int64_t count, int32_t n);

/* Host-only helper: the sum of the FP32 squares v[i] * v[i] of `count` values (BF16 values given
 * as FP32, in host memory), rounded to FP32 exactly as the kernels' rare exact path rounds a row
 * or head sum of squares ("Sandwich-Norm": RMSNorm in FP32): in 128-bit fixed point scaled to the
 * largest square, then rounded once to nearest even.  NaN if a square is NaN, +inf if one is
 * infinite or the sum overflows, 0 if all are zero.  The result is the exact rounding unless some
 * square lies more than 2^88 below the largest and the sum falls within 2^-98 (relative) of a
 * rounding boundary.  Returns BEAM_ERR_INVALID_ARG for count < 0, count > 16384 or NULL arrays. */
BEAM_API int beam_exact_square_sum(const float *v, int64_t count, float *out);

/* Host-only helper: the FP32 sigmoid that beam_grouped_topk_fwd ranks experts by,
 * sigma(z) = 1 / (1 + RN32(exp(-z))) (FP32 add, IEEE division, exp rounded once to FP32: FP32
 * pair arithmetic with an FP64 pair fallback near rounding boundaries), for `count` values in
 * host memory.  NaN stays NaN.  Returns BEAM_ERR_INVALID_ARG for count < 0 or NULL arrays. */
BEAM_API int beam_routing_sigmoid(const float *z, float *out, int64_t count);

/* Host-only helper: the FP32 cosine and sine that beam_qk_norm_rope_fwd uses for an FP32 rotary
 * angle, for `count` angles in host memory.  Each value is the FP32 rounding of the exact
 * cos / sin of the FP32 angle (except in rare near-tie cases), computed in FP32 pair arithmetic
 * (Cody-Waite reduction, Dekker products, Taylor series).  Angles must satisfy |a| < 2^24;
 * others give NaN outputs and BEAM_ERR_INVALID_ARG.  Returns BEAM_ERR_INVALID_ARG for NULL
 * arrays (count > 0) or count < 0. */
BEAM_API int beam_rope_cos_sin(const float *angle, float *cos_out, float *sin_out, int64_t count);

/* Sublayer boundary: post-RMSNorm -> depth-scaled residual add -> next pre-RMSNorm, per token.
 *
 * Defined by [vLLM] "MoE und Residual-Stream" (bullets "Sandwich-Norm": an RMSNorm before and
 * after every sublayer; "Tiefenskalierte Residuen": the n-th residual add is
 * h <- sqrt((n-1)/n) h + x/sqrt(n)), [vLLM] "Agentengetriebene Optimierung" change 1 (the three
 * steps fused at each of the 104 boundaries, FP32 math, the reference BF16 rounding points) and
 * [SGL] "三明治归一化与深度缩放残差" (both scaled operands rounded to BF16 before the add).
 *
 * For every token t (row of H elements), with m(v) = fp32(sum_j fp32(v_j^2)) / H:
 *   r     = 1 / sqrt(m(x) + eps)
 *   xhat  = bf16((x * r) * w_post)                      post-norm of the sublayer output
 *   a     = bf16(alpha * h),  b = bf16(xhat / s),  h' = bf16(a + b)
 *   r'    = 1 / sqrt(m(h') + eps)
 *   y     = bf16((h' * r') * w_pre)                     pre-norm of the next sublayer
 * with alpha, s from beam_residual_scales(n).  The sum of squares is formed to within ~1e-11
 * relative of its exact value before its single FP32 rounding.
 *
 *   h_out  [T, H] bf16  out: h'              (may be the same buffer as h_in)
 *   y_out  [T, H] bf16  out: y               (may be the same buffer as x_in)
 *   h_in   [T, H] bf16  residual stream before the add
 *   x_in   [T, H] bf16  sublayer output (before its post-norm)
 *   w_post [H]    bf16  post-norm weight of the sublayer;  w_pre [H] bf16 next pre-norm weight
 *   T >= 0 tokens; H hidden size, a multiple of 8 in [8, 16384]; n >= 1 residual index;
 *   eps >= 0 and finite;
 *   rstd_out [T, 2] fp32 or NULL: (r, r') per token.
 * Rows are contiguous (row stride H). */
BEAM_API int beam_boundary_fwd(void *h_out, void *y_out, const void *h_in, const void *x_in,
                      const void *w_post, const void *w_pre, int64_t T, int32_t H, int32_t n,
                      float eps, float *rstd_out, cudaStream_t stream);

/* MoE top-K combine fused ahead of the boundary chain.
 *
 * [vLLM] "MoE und Residual-Stream", bullet "MoE im DeepSeek-V3-Stil" (top-8 experts, the
 * renormalised weights scaled by 2.5); [vLLM] "Agentengetriebene Optimierung" change 3 (the
 * boundary kernel also combines the top-8 expert outputs); [SGL] "稠密层与分组 MoE 路由"
 * (routing coefficients kept in FP32 and the scale applied in the combine) and its
 * kernel-fusion paragraph (expert sum, routing scale and BF16 rounding in one place).
 *
 * Per token: c_k = fp32(topk_w[t,k] * routed_scaling);
 *   x_j = bf16(acc), acc = fma(c_{K-1}, e_{K-1,j}, ... fma(c_1, e_{1,j}, fma(c_0, e_{0,j}, +0)))
 * i.e. one FP32 fused multiply-add per slot in slot order 0..K-1; then exactly the
 * beam_boundary_fwd chain on x.
 *
 *   expert_out [T, K, H] bf16  the K selected experts' outputs per token, slot-major per token
 *   topk_w     [T, K]    fp32  renormalised routing weights (renormalisation is the caller's)
 *   routed_scaling             finite (2.5 for Beam);  K in [1, 16]
 *   other arguments as beam_boundary_fwd (h_out may equal h_in; no other overlap). */
BEAM_API int beam_moe_combine_boundary_fwd(void *h_out, void *y_out, const void *h_in,
                                  const void *expert_out, const float *topk_w,
                                  float routed_scaling, const void *w_post, const void *w_pre,
                                  int64_t T, int32_t H, int32_t K, int32_t n, float eps,
                                  float *rstd_out, cudaStream_t stream);

/* Tensor-parallel all-reduce of the sublayer output fused ahead of the boundary chain.
 *
 * [vLLM] "Agentengetriebene Optimierung", change 3 (both TP all-reduces of every layer run
 * inside the norm kernel); [SGL] kernel-fusion paragraph (the all-reduce, the output norm, the
 * scaled residual add and the next layer's input norm fused in one kernel).
 *
 * Under tensor parallelism over P ranks each rank holds a partial sublayer output x_p.  Per
 * token and element, in rank order (FP32 adds, starting from rank 0's value, one rounding):
 *   x_j = bf16( (((x_{0,j} + x_{1,j}) + x_{2,j}) + ...) + x_{P-1,j} )
 * then exactly the beam_boundary_fwd chain on x.  With P = 1 the call is beam_boundary_fwd on
 * x_parts[0].  Every rank that runs it on the same partials gets bit-identical h' and y.
 *
 *   x_parts  host array of P device pointers, each a [T, H] bf16 partial (16-byte aligned,
 *            rows contiguous); the same buffer may appear more than once
 *   P        in [1, 16]
 *   other arguments as beam_boundary_fwd.  h_out may be the same buffer as h_in, and y_out may be
 *   the same buffer as one of the partials; no other overlap.
 * This call reads the P partials from this GPU's memory.  Gathering the other ranks' partials
 * (peer copies, or peer-mapped buffers passed here directly) is the caller's. */
BEAM_API int beam_allreduce_boundary_fwd(void *h_out, void *y_out, const void *h_in,
                                         const void *const *x_parts, int32_t P,
                                         const void *w_post, const void *w_pre, int64_t T,
                                         int32_t H, int32_t n, float eps, float *rstd_out,
                                         cudaStream_t stream);

/* Per-head Q/K RMSNorm fused with rotary embedding (sliding-window layers), in place.
 *
 * [vLLM] "Attention", bullets "GQA mit Per-Head-Q/K-Norm" (48 query heads, 8 KV heads, head
 * dimension 128; Q and K RMS-normalised per head before RoPE or SSMax) and "Hybride
 * Sliding-Window- und NoPE-Schichten" (RoPE on the sliding-window layers); [SGL] kernel-fusion
 * paragraph (sliding-window layers fuse the Q/K norm with RoPE).
 *
 * Per token t and head (row v of 128 elements, weight w = wq for Q heads, wk for K heads):
 *   r = 1 / sqrt(m(v) + eps);  qhat_d = (v_d * r) * w_d   (FP32, not rounded)
 * m(v) = fp32(sum of the FP32 squares) / 128, the sum rounded as the exact sum would be (the
 * rotation can cancel, so an FP32 ulp of r could otherwise move an output by more than one
 * BF16 ulp).
 *   angle_i = fp32(fp32(pos[t]) * inv_freq_i),  inv_freq_i = fp32(theta^(-2i/128)), i < 64
 *   out_i    = bf16( fp32(qhat_i * cos_i)    - fp32(qhat_{i+64} * sin_i) )
 *   out_{i+64} = bf16( fp32(qhat_{i+64} * cos_i) + fp32(qhat_i * sin_i) )
 * cos_i / sin_i are the FP32 roundings of the exact cosine and sine of the FP32 angle
 * (beam_rope_cos_sin) when |angle_i| < 2^24 (always, for positions < 2^24 and theta >= 1);
 * larger angles use CUDA's sincosf (within 2 FP32 ulps).
 *
 *   q [T, n_q_heads, 128] bf16 in place, row t at q + t*q_row_stride (elements)
 *   k [T, n_kv_heads, 128] bf16 in place, row t at k + t*k_row_stride
 *   wq, wk [128] bf16 norm weights (shared by all heads of Q, resp. K)
 *   pos [T] int64, 0-based positions >= 0 (converted to FP32; exact below 2^24)
 *   n_q_heads, n_kv_heads >= 0 with n_q_heads + n_kv_heads in [1, 1024]; head_dim must be 128
 *   (else BEAM_ERR_UNSUPPORTED); eps >= 0; theta > 0.  q (k) may be NULL when n_q_heads
 *   (n_kv_heads) is 0.  Strides >= the row length and multiples of 8, so Q and K may be views
 *   into one packed QKV(+gate) projection output; q and k rows must not overlap. */
BEAM_API int beam_qk_norm_rope_fwd(void *q, void *k, int64_t q_row_stride, int64_t k_row_stride,
                          const void *wq, const void *wk, const int64_t *pos, int64_t T,
                          int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, float eps,
                          float theta, cudaStream_t stream);

/* Per-head Q/K RMSNorm fused with the SSMax query scale (NoPE layers), in place.
 *
 * [vLLM] "Attention", bullet "SSMax auf NoPE-Schichten" (each query scaled by (1 + p/2048)^0.1,
 * p the 1-based position); [SGL] "稠密层与分组 MoE 路由", SSMax paragraph (after the Q/K norm,
 * the query at 0-based position p is scaled by (1 + (p+1)/2048)^0.1).
 *
 * Q heads: out = bf16( ((v * r) * wq) * sigma_t ),  sigma_t = powf(1 + fp32(pos[t]+1) / base, expo)
 * (CUDA's powf, within a few FP32 ulps of the exact value);  K heads: out = bf16( (v * r) * wk )
 * (no scale).  r as for RoPE, except that the head sum of squares is a plain FP32 sum in a fixed
 * order: the outputs only scale with r, so an FP32 ulp moves them by at most one BF16 ulp.
 * Arguments as beam_qk_norm_rope_fwd; ssmax_base > 0 (2048), ssmax_exp finite (0.1). */
BEAM_API int beam_qk_norm_ssmax_fwd(void *q, void *k, int64_t q_row_stride, int64_t k_row_stride,
                           const void *wq, const void *wk, const int64_t *pos, int64_t T,
                           int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim, float eps,
                           float ssmax_base, float ssmax_exp, cudaStream_t stream);

/* The Q/K calls above fused with the KV-cache write of the same tokens.
 *
 * [vLLM] "MoE und Residual-Stream", change 6 (the Q/K-norm and RoPE kernel also writes K and V
 * into the KV cache, so no separate cache-write kernel runs) and the serving command's FP8 KV
 * cache; [vLLM] "Attention", bullet "Kleiner KV-Cache" (only the full-attention layers keep the
 * whole sequence); [SGL] "目标模型与草稿模型 KV 的统一内存" (KV writes go to each token's physical
 * slot).
 *
 * Q and K are normalised (and rotated, or scaled) in place exactly as by beam_qk_norm_rope_fwd /
 * beam_qk_norm_ssmax_fwd.  In the same pass, for each token t whose slot s = slot_mapping[t]
 * lies in [0, num_slots):
 *   k_cache[s, h, :] = K'[t, h, :]  (the stored, normalised K)   v_cache[s, h, :] = V[t, h, :]
 * as BF16 (cache_dtype 0: the bits) or FP8 E4M3 (cache_dtype 1: fp8(value / scale), FP32
 * division, round to nearest even, saturating to +-448, NaN to a NaN code).  Tokens with a
 * negative (padding) or out-of-range slot write no cache row.  Slots of one call must be
 * distinct; if two tokens share one, which row lands is unspecified.
 *
 *   v [T, n_kv_heads, 128] bf16, row t at v + t*v_row_stride (elements; >= n_kv_heads*128,
 *     multiple of 8, 16-byte aligned); read only
 *   slot_mapping [T] int64;  k_cache, v_cache [num_slots, n_kv_heads, 128], contiguous, 2 bytes
 *     per element (16-byte aligned) for BF16, 1 byte (8-byte aligned) for FP8; must not overlap
 *     each other or the other arguments
 *   k_scale, v_scale: finite and > 0 for FP8 (ignored for BF16)
 * BEAM_ERR_UNSUPPORTED for any other cache_dtype; with n_kv_heads == 0 nothing is cached and
 * the cache arguments may be NULL.  Other arguments and checks as the calls above. */
BEAM_API int beam_qk_norm_rope_kv_fwd(void *q, void *k, int64_t q_row_stride, int64_t k_row_stride,
                             const void *v, int64_t v_row_stride, const void *wq, const void *wk,
                             const int64_t *pos, const int64_t *slot_mapping, void *k_cache,
                             void *v_cache, int64_t num_slots, int32_t cache_dtype, float k_scale,
                             float v_scale, int64_t T, int32_t n_q_heads, int32_t n_kv_heads,
                             int32_t head_dim, float eps, float theta, cudaStream_t stream);

BEAM_API int beam_qk_norm_ssmax_kv_fwd(void *q, void *k, int64_t q_row_stride, int64_t k_row_stride,
                              const void *v, int64_t v_row_stride, const void *wq, const void *wk,
                              const int64_t *pos, const int64_t *slot_mapping, void *k_cache,
                              void *v_cache, int64_t num_slots, int32_t cache_dtype, float k_scale,
                              float v_scale, int64_t T, int32_t n_q_heads, int32_t n_kv_heads,
                              int32_t head_dim, float eps, float ssmax_base, float ssmax_exp,
                              cudaStream_t stream);

/* DeepSeek-V3-style grouped top-k routing: the step that produces the MoE combine's inputs.
 *
 * [vLLM] "MoE und Residual-Stream", bullet "MoE im DeepSeek-V3-Stil" (256 routed experts,
 * routed as in DeepSeek-V3: sigmoid scores plus a correction bias choose the best 4 of 8 expert
 * groups, then the top 8 experts; the renormalised weights are scaled by 2.5) and bullet
 * "FP32-Router" (logits in FP32); [SGL] "稠密层与分组 MoE 路由" (grouped top-k from the sigmoid
 * scores and the expert correction bias; FP32 routing coefficients, the scaling applied in the
 * combine).
 *
 * Per token t, with s_e = 1 / (1 + RN32(exp(-logit_e))) (as beam_routing_sigmoid) and the choice
 * score c_e = fp32(s_e + bias_e):
 *   - each of the 8 groups of 32 consecutive experts scores fp32(c_first + c_second), its two
 *     best choice scores (DeepSeek-V3's group rule); the 4 best groups stay eligible;
 *   - topk_ids[t, k], k < 8: the 8 best eligible experts by c, best first;
 *   - topk_w[t, k] = s_{id_k} / S, S the FP32 sum of those 8 scores in slot order (IEEE
 *     division): renormalised, not yet scaled -- beam_moe_combine_boundary_fwd applies the
 *     routed scaling (2.5).
 * Ranking: larger first; NaN below every number; ties to the lower index.  Because every
 * sigmoid is the correctly rounded FP32 value, the choice is bit-reproducible.
 *
 *   logits [T, 256] fp32 (16-byte aligned rows), bias [256] fp32 (16-byte aligned)
 *   topk_ids [T, 8] int32, topk_w [T, 8] fp32 (4-byte aligned)
 * n_experts, n_groups, topk_groups, top_k must be 256, 8, 4, 8 (BEAM_ERR_UNSUPPORTED otherwise). */
BEAM_API int beam_grouped_topk_fwd(int32_t *topk_ids, float *topk_w, const float *logits,
                                   const float *bias, int64_t T, int32_t n_experts,
                                   int32_t n_groups, int32_t topk_groups, int32_t top_k,
                                   cudaStream_t stream);

/* Sigmoid attention-output gate, before the output projection.
 *
 * [vLLM] "Attention", bullet "Sigmoid-Output-Gate" (each head's output times
 * sigma(gate + bias) with a learned per-head bias; a head can be switched off token by token);
 * [SGL] "混合注意力与输出门控" and the kernel-fusion paragraph (bias add, sigmoid and multiply
 * fused in one kernel).
 *
 * out[t, h*D + d] = bf16( attn * (1 / (1 + expf(-z))) ),  z = fp32(gate[t, h*D + d] + bias[h]),
 * with CUDA's full-accuracy expf, an FP32 add and the hardware reciprocal (within one FP32 ulp;
 * exact for 1/2 and 1/inf).  The output scales with the sigmoid, so these few FP32 ulps move it
 * by at most one BF16 ulp.
 *
 *   out, attn, gate  [T, n_heads*head_dim] bf16 rows at the given strides (elements, >= the row
 *   length, multiples of 8); out may be the same buffer as attn (same stride) for in-place use.
 *   bias [n_heads] fp32 (+-inf allowed: -inf switches a head off, +inf passes it through).
 *   n_heads in [1, 1024]; head_dim a multiple of 8 in [8, 1024]. */
BEAM_API int beam_attn_gate_fwd(void *out, const void *attn, const void *gate, const float *bias,
                       int64_t T, int32_t n_heads, int32_t head_dim, int64_t attn_row_stride,
                       int64_t gate_row_stride, int64_t out_row_stride, cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* BEAM_BOUNDARY_H */
