/*
 * beam_oracle.c -- plain, slow CPU oracle for the Beam sublayer-boundary path.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference leg may load this library.  It shares no code with the
 * CUDA library (no headers, helpers or tables); the two meet only on the seeded inputs.
 *
 * Every function works one token at a time, in program order, in FP32 arithmetic with the BF16
 * round-to-nearest-even points the pages state.  Two steps are computed as their exact values
 * rounded once, so the oracle is the exact side of every comparison:
 *   - a row's sum of squares is summed exactly (integer fixed point) and rounded once to FP32;
 *   - exp / cos / sin / pow are evaluated in double and rounded once to FP32.
 * Build with -ffp-contract=off: a contracted multiply-add would change the FP32 rounding steps.
 *
 * Pages cited (titles as printed):
 *   [vLLM]  "Serving Reflection Beam auf vLLM ab Tag 0"
 *   [SGL]   "SGLang 支撑编程模型 Beam 生产部署"
 *
 * Parity pins: every function here is pinned by the CPU tests (tests/test_oracle_*.py) against
 * closed forms, invariants and library routines; none is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* ------------------------------------------------------------------------------------------ */
/* BF16                                                                                        */
/* ------------------------------------------------------------------------------------------ */

/* FP32 -> BF16 with IEEE round-to-nearest-even.  NaN stays NaN (quiet bit set); overflow past
 * the largest finite BF16 goes to infinity; subnormals round like any other value.
 * [SGL] "三明治归一化与深度缩放残差": both scaled residual operands are rounded to the
 * activation type (BF16) before the add; RNE is the IEEE default rounding. */
uint16_t orc_bf16_rne(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7fffffffu) > 0x7f800000u)          /* NaN: keep sign and payload top, force quiet */
        return (uint16_t)((u >> 16) | 0x0040u);
    uint32_t lsb = (u >> 16) & 1u;                /* ties go to the even neighbour */
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* value of x after a BF16 rounding, as FP32 */
static float bf16_round(float x) { return orc_bf16_to_f32(orc_bf16_rne(x)); }

void orc_bf16_rne_array(const float *in, uint16_t *out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = orc_bf16_rne(in[i]);
}

/* ------------------------------------------------------------------------------------------ */
/* RMSNorm scale                                                                               */
/* ------------------------------------------------------------------------------------------ */

/* Exact sum of non-negative FP32 terms, rounded once to FP32 with round-to-nearest-even.
 * Every finite FP32 value is an integer multiple of 2^-149 (the smallest subnormal), so the
 * terms are added exactly as integers in a 384-bit fixed-point accumulator (a Kulisch
 * accumulator: bit i of the integer is worth 2^(i-149)); the result is rounded once.  A NaN term
 * makes the sum NaN, an infinite term (and no NaN) makes it +inf. */
typedef struct {
    uint64_t limb[6];
    int nan, inf;
} exact_sum;

static void exact_sum_init(exact_sum *a)
{
    memset(a, 0, sizeof *a);
}

static void exact_sum_add(exact_sum *a, float t)
{
    uint32_t u;
    memcpy(&u, &t, sizeof u);
    uint32_t e = (u >> 23) & 0xffu;
    uint64_t m = u & 0x7fffffu;
    if (e == 0xffu) {
        if (m)
            a->nan = 1;
        else
            a->inf = 1;
        return;
    }
    if (e)
        m |= 0x800000u;      /* normal: t = m * 2^(e - 150) = m * 2^(e - 1) * 2^-149 */
    else
        e = 1;               /* subnormal: t = m * 2^-149 */
    uint32_t p = e - 1;      /* bit position of m's lowest bit */
    uint32_t li = p / 64, sh = p % 64;
    unsigned __int128 v = (unsigned __int128)m << sh;
    uint64_t lo = (uint64_t)v, hi = (uint64_t)(v >> 64);
    uint64_t before = a->limb[li];
    a->limb[li] += lo;
    uint64_t carry = a->limb[li] < before;
    for (uint32_t k = li + 1; k < 6 && (hi || carry); ++k) {
        before = a->limb[k];
        a->limb[k] += hi + carry;
        carry = (a->limb[k] < before) || (carry && hi + carry == 0);
        hi = 0;
    }
}

static int exact_sum_bit(const exact_sum *a, int i)
{
    return i < 0 ? 0 : (int)((a->limb[i / 64] >> (i % 64)) & 1u);
}

static float exact_sum_round(const exact_sum *a)
{
    if (a->nan)
        return NAN;
    if (a->inf)
        return INFINITY;
    int top = -1;
    for (int i = 6 * 64 - 1; i >= 0; --i)
        if (exact_sum_bit(a, i)) {
            top = i;
            break;
        }
    if (top < 0)
        return 0.0f;
    if (top < 24)  /* fewer than 25 significant bits: exactly representable */
        return ldexpf((float)a->limb[0], -149);
    uint32_t mant = 0;
    for (int i = top; i > top - 24; --i)
        mant = (mant << 1) | (uint32_t)exact_sum_bit(a, i);
    int half = exact_sum_bit(a, top - 24), sticky = 0;
    for (int i = top - 25; i >= 0 && !sticky; --i)
        sticky = exact_sum_bit(a, i);
    if (half && (sticky || (mant & 1u))) {
        mant += 1;
        if (mant == (1u << 24)) {
            mant >>= 1;
            top += 1;
        }
    }
    return ldexpf((float)mant, (top - 23) - 149);  /* exact, or +inf past the FP32 range */
}

/* r = 1 / sqrt(mean_j v_j^2 + eps).
 * Each square is an FP32 product; their exact sum is rounded once to FP32; the mean is that FP32
 * sum divided by the length in FP32; then FP32 add, IEEE sqrt, IEEE div.
 * [vLLM] "MoE und Residual-Stream", bullet "Sandwich-Norm": an RMSNorm before and after every
 * sublayer; [vLLM] "Agentengetriebene Optimierung", change 1: FP32 math. */
static float rms_inv(const float *v, int32_t len, float eps)
{
    exact_sum acc;
    exact_sum_init(&acc);
    for (int32_t j = 0; j < len; ++j) {
        float sq = v[j] * v[j];
        exact_sum_add(&acc, sq);
    }
    float ms = exact_sum_round(&acc);
    float mean = ms / (float)len;
    return 1.0f / sqrtf(mean + eps);
}

/* Test hook: the exactly rounded FP32 sum of `count` non-negative FP32 terms. */
float orc_exact_sum_f32(const float *terms, int64_t count)
{
    exact_sum acc;
    exact_sum_init(&acc);
    for (int64_t i = 0; i < count; ++i)
        exact_sum_add(&acc, terms[i]);
    return exact_sum_round(&acc);
}

/* ------------------------------------------------------------------------------------------ */
/* Sublayer boundary: post-RMSNorm -> depth-scaled residual add -> next pre-RMSNorm            */
/* ------------------------------------------------------------------------------------------ */

/* Coefficients of the n-th residual add, h <- sqrt((n-1)/n) * h + x / sqrt(n), as FP32.
 * [vLLM] "MoE und Residual-Stream", bullet "Tiefenskalierte Residuen". */
void orc_residual_scales(int32_t n, float *alpha, float *s)
{
    *alpha = (float)sqrt((double)(n - 1) / (double)n);
    *s = (float)sqrt((double)n);
}

/* One token of the boundary chain on an FP32 copy of the sublayer output xf[H].
 *   a1  r  = rms_inv(x);            xhat_j = bf16((x_j * r) * wpost_j)
 *   a2  a_j = bf16(alpha * h_j);    b_j = bf16(xhat_j / s);    h'_j = bf16(a_j + b_j)
 *   a3  r' = rms_inv(h');           y_j = bf16((h'_j * r') * wpre_j)
 * [vLLM] "Agentengetriebene Optimierung", change 1 (post-norm, scaled add and next pre-norm in
 * one pass, FP32 math, the reference BF16 rounding points); [SGL] "三明治归一化与深度缩放残差"
 * (both scaled operands rounded to BF16 before the add; the normalised branch result is a
 * materialised BF16 tensor in the unfused path). */
static void boundary_token(uint16_t *h_out, uint16_t *y_out, const uint16_t *h_in,
                           const float *xf, const uint16_t *w_post, const uint16_t *w_pre,
                           int32_t H, float alpha, float s, float eps, float *rstd2,
                           float *work /* [2H] */)
{
    float *xhat = work;
    float *hp = work + H;

    float r1 = rms_inv(xf, H, eps);
    for (int32_t j = 0; j < H; ++j) {
        float t = xf[j] * r1;
        xhat[j] = bf16_round(t * orc_bf16_to_f32(w_post[j]));
    }
    for (int32_t j = 0; j < H; ++j) {
        float a = bf16_round(alpha * orc_bf16_to_f32(h_in[j]));
        float b = bf16_round(xhat[j] / s);
        hp[j] = bf16_round(a + b);
    }
    float r2 = rms_inv(hp, H, eps);
    for (int32_t j = 0; j < H; ++j) {
        float t = hp[j] * r2;
        y_out[j] = orc_bf16_rne(t * orc_bf16_to_f32(w_pre[j]));
        h_out[j] = orc_bf16_rne(hp[j]);
    }
    if (rstd2) {
        rstd2[0] = r1;
        rstd2[1] = r2;
    }
}

/* h_in, x_in, h_out, y_out: [T, H] BF16 bit patterns, rows contiguous.  rstd_out: [T, 2] or NULL.
 * work: caller scratch of 3*H floats.  Outputs must not alias inputs. */
void orc_boundary(uint16_t *h_out, uint16_t *y_out, const uint16_t *h_in, const uint16_t *x_in,
                  const uint16_t *w_post, const uint16_t *w_pre, int64_t T, int32_t H, int32_t n,
                  float eps, float *rstd_out, float *work)
{
    float alpha, s;
    orc_residual_scales(n, &alpha, &s);
    float *xf = work + 2 * (int64_t)H;
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < H; ++j)
            xf[j] = orc_bf16_to_f32(x_in[t * H + j]);
        boundary_token(h_out + t * H, y_out + t * H, h_in + t * H, xf, w_post, w_pre, H, alpha,
                       s, eps, rstd_out ? rstd_out + 2 * t : 0, work);
    }
}

/* ------------------------------------------------------------------------------------------ */
/* MoE top-K combine fused ahead of the boundary                                               */
/* ------------------------------------------------------------------------------------------ */

/* x_j = bf16( sum_k c_k * e_{k,j} ),  c_k = fp32(w_k * routed_scaling).
 * The sum runs in slot order k = 0..K-1, one FP32 fused multiply-add per slot, from +0.
 * Then the boundary chain on x.
 * [vLLM] "MoE und Residual-Stream", bullet "MoE im DeepSeek-V3-Stil" (top-8, renormalised
 * weights scaled by 2.5); [vLLM] "Agentengetriebene Optimierung", change 3 (the boundary kernel
 * also combines the top-8 expert outputs); [SGL] "稠密层与分组 MoE 路由" (FP32 routing
 * coefficients, scaling factor applied in the combine); [SGL] kernel-fusion paragraph (local
 * expert sum, routing scale and BF16 rounding fused).
 * expert_out: [T, K, H]; topk_w: [T, K] FP32; x_out: [T, H] or NULL (the combined x, for tests). */
void orc_moe_combine_boundary(uint16_t *h_out, uint16_t *y_out, const uint16_t *h_in,
                              const uint16_t *expert_out, const float *topk_w,
                              float routed_scaling, const uint16_t *w_post,
                              const uint16_t *w_pre, int64_t T, int32_t H, int32_t K, int32_t n,
                              float eps, float *rstd_out, uint16_t *x_out, float *work)
{
    float alpha, s;
    orc_residual_scales(n, &alpha, &s);
    float *xf = work + 2 * (int64_t)H;
    float c[64];
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t k = 0; k < K; ++k)
            c[k] = topk_w[t * K + k] * routed_scaling;
        const uint16_t *e = expert_out + t * (int64_t)K * H;
        for (int32_t j = 0; j < H; ++j) {
            float acc = 0.0f;
            for (int32_t k = 0; k < K; ++k)
                acc = fmaf(c[k], orc_bf16_to_f32(e[(int64_t)k * H + j]), acc);
            xf[j] = bf16_round(acc);
            if (x_out)
                x_out[t * H + j] = orc_bf16_rne(acc);
        }
        boundary_token(h_out + t * H, y_out + t * H, h_in + t * H, xf, w_post, w_pre, H, alpha,
                       s, eps, rstd_out ? rstd_out + 2 * t : 0, work);
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Tensor-parallel all-reduce of the sublayer output fused ahead of the boundary               */
/* ------------------------------------------------------------------------------------------ */

/* Under tensor parallelism over P ranks each rank holds a partial sublayer output x_p (BF16);
 * the sublayer output is their sum.  Per element, in rank order:
 *   s_0 = x_{0,j};   s_p = fp32(s_{p-1} + x_{p,j}) for p = 1..P-1;   x_j = bf16(s_{P-1})
 * (FP32 adds, one BF16 rounding), then the boundary chain on x.  With P = 1 this is the plain
 * boundary on x_0.
 * [vLLM] "Agentengetriebene Optimierung", change 3 (both TP all-reduces of a layer run inside
 * the norm kernel); [SGL] kernel-fusion paragraph (all-reduce, output norm, scaled residual add
 * and the next layer's input norm fused).  Neither page states the accumulation order; rank
 * order in FP32 is the plainest reading of "FP32 math" ([vLLM] change 1).
 * parts: [P, T, H] BF16 (rank p's partial at parts + p*T*H); x_out: [T, H] or NULL. */
void orc_allreduce_boundary(uint16_t *h_out, uint16_t *y_out, const uint16_t *h_in,
                            const uint16_t *parts, int32_t P, const uint16_t *w_post,
                            const uint16_t *w_pre, int64_t T, int32_t H, int32_t n, float eps,
                            float *rstd_out, uint16_t *x_out, float *work)
{
    float alpha, s;
    orc_residual_scales(n, &alpha, &s);
    float *xf = work + 2 * (int64_t)H;
    const int64_t plane = T * (int64_t)H;
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t j = 0; j < H; ++j) {
            float acc = orc_bf16_to_f32(parts[t * H + j]);
            for (int32_t p = 1; p < P; ++p)
                acc = acc + orc_bf16_to_f32(parts[p * plane + t * H + j]);
            xf[j] = bf16_round(acc);
            if (x_out)
                x_out[t * H + j] = orc_bf16_rne(acc);
        }
        boundary_token(h_out + t * H, y_out + t * H, h_in + t * H, xf, w_post, w_pre, H, alpha,
                       s, eps, rstd_out ? rstd_out + 2 * t : 0, work);
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Per-head Q/K RMSNorm fused with RoPE (sliding-window layers) or SSMax (NoPE layers)          */
/* ------------------------------------------------------------------------------------------ */

/* qhat_d = (v_d * r) * w_d in FP32, no rounding, r = rms_inv over the head.
 * [vLLM] "Attention", bullet "GQA mit Per-Head-Q/K-Norm": Q and K are RMS-normalised per head
 * before RoPE or SSMax; [SGL] "混合注意力与输出门控". */
static void head_norm(float *qhat, const uint16_t *v, const uint16_t *w, int32_t D, float eps,
                      float *tmp)
{
    for (int32_t d = 0; d < D; ++d)
        tmp[d] = orc_bf16_to_f32(v[d]);
    float r = rms_inv(tmp, D, eps);
    for (int32_t d = 0; d < D; ++d)
        qhat[d] = (tmp[d] * r) * orc_bf16_to_f32(w[d]);
}

/* Rotary frequencies of the half-rotation convention: inv_freq_i = fp32(theta^(-2i/D)). */
void orc_rope_inv_freq(float theta, int32_t D, float *inv_freq)
{
    for (int32_t i = 0; i < D / 2; ++i)
        inv_freq[i] = (float)pow((double)theta, -2.0 * (double)i / (double)D);
}

/* In place on q rows [T, nq, D] (row stride q_stride elements) and k rows [T, nk, D].
 * Per token: angle_i = fp32(fp32(pos) * inv_freq_i); c_i, s_i = cos, sin of that FP32 angle
 * (double, rounded to FP32).  Per head, half rotation over the pairs (i, i + D/2):
 *   out_i       = bf16( fp32(qhat_i * c_i) - fp32(qhat_{i+D/2} * s_i) )
 *   out_{i+D/2} = bf16( fp32(qhat_{i+D/2} * c_i) + fp32(qhat_i * s_i) )
 * [vLLM] "Attention", bullet "Hybride Sliding-Window- und NoPE-Schichten" (RoPE on the 43
 * sliding-window layers); [SGL] kernel-fusion paragraph (Q/K norm fused with RoPE). */
void orc_qk_norm_rope(uint16_t *q, uint16_t *k, int64_t q_stride, int64_t k_stride,
                      const uint16_t *wq, const uint16_t *wk, const int64_t *pos, int64_t T,
                      int32_t nq, int32_t nk, int32_t D, float eps, float theta, float *work)
{
    int32_t half = D / 2;
    float *inv_freq = work;           /* [D/2] */
    float *cs = work + half;          /* [D/2] */
    float *sn = work + 2 * half;      /* [D/2] */
    float *qhat = work + 3 * half;    /* [D] */
    float *tmp = work + 3 * half + D; /* [D] */
    orc_rope_inv_freq(theta, D, inv_freq);
    for (int64_t t = 0; t < T; ++t) {
        float p = (float)pos[t];
        for (int32_t i = 0; i < half; ++i) {
            float ang = p * inv_freq[i];
            cs[i] = (float)cos((double)ang);
            sn[i] = (float)sin((double)ang);
        }
        for (int32_t hd = 0; hd < nq + nk; ++hd) {
            uint16_t *row = hd < nq ? q + t * q_stride + (int64_t)hd * D
                                    : k + t * k_stride + (int64_t)(hd - nq) * D;
            const uint16_t *w = hd < nq ? wq : wk;
            head_norm(qhat, row, w, D, eps, tmp);
            for (int32_t i = 0; i < half; ++i) {
                float lo = qhat[i] * cs[i] - qhat[i + half] * sn[i];
                float hi = qhat[i + half] * cs[i] + qhat[i] * sn[i];
                row[i] = orc_bf16_rne(lo);
                row[i + half] = orc_bf16_rne(hi);
            }
        }
    }
}

/* SSMax query scale for a 0-based position: fp32((1 + (pos + 1) / base) ^ expo).
 * [vLLM] "Attention", bullet "SSMax auf NoPE-Schichten": (1 + p/2048)^0.1 with p 1-based;
 * [SGL] "稠密层与分组 MoE 路由", SSMax paragraph: the same with a 0-based p as (1+(p+1)/2048)^0.1. */
float orc_ssmax_scale(int64_t pos, float base, float expo)
{
    double p1 = (double)pos + 1.0;
    return (float)pow(1.0 + p1 / (double)base, (double)expo);
}

/* In place.  Q: out = bf16( ((q * r) * wq) * ssmax_scale(pos) );  K: out = bf16( (k * r) * wk ).
 * The scale multiplies queries only, after their norm. */
void orc_qk_norm_ssmax(uint16_t *q, uint16_t *k, int64_t q_stride, int64_t k_stride,
                       const uint16_t *wq, const uint16_t *wk, const int64_t *pos, int64_t T,
                       int32_t nq, int32_t nk, int32_t D, float eps, float base, float expo,
                       float *work)
{
    float *qhat = work;
    float *tmp = work + D;
    for (int64_t t = 0; t < T; ++t) {
        float sc = orc_ssmax_scale(pos[t], base, expo);
        for (int32_t hd = 0; hd < nq + nk; ++hd) {
            int is_q = hd < nq;
            uint16_t *row = is_q ? q + t * q_stride + (int64_t)hd * D
                                 : k + t * k_stride + (int64_t)(hd - nq) * D;
            head_norm(qhat, row, is_q ? wq : wk, D, eps, tmp);
            for (int32_t d = 0; d < D; ++d)
                row[d] = orc_bf16_rne(is_q ? qhat[d] * sc : qhat[d]);
        }
    }
}

/* ------------------------------------------------------------------------------------------ */
/* DeepSeek-V3-style grouped top-k routing (the step that produces the combine's inputs)        */
/* ------------------------------------------------------------------------------------------ */

/* FP32 sigmoid: 1 / (1 + e) with e = exp(-z) rounded once to FP32 (evaluated in long double),
 * then an FP32 add and an IEEE FP32 division.  exp(-z) overflowing gives e = inf and 0. */
float orc_sigmoid_f32(float z)
{
    float e = (float)expl(-(long double)z);
    return 1.0f / (1.0f + e);
}

void orc_sigmoid_array(const float *z, float *out, int64_t count)
{
    for (int64_t i = 0; i < count; ++i)
        out[i] = orc_sigmoid_f32(z[i]);
}

/* FP32 rounding of exp(x), evaluated in long double (test hook). */
float orc_exp_f32(float x) { return (float)expl((long double)x); }

/* Routing order: a number ranks above NaN; between numbers the larger value; ties (and NaN
 * against NaN) go to the lower index. */
static int ranks_above(float a, int32_t ia, float b, int32_t ib)
{
    int na = isnan(a), nb = isnan(b);
    if (na != nb)
        return nb;
    if (!na && a != b)
        return a > b;
    return ia < ib;
}

/* Per token: s_e = sigmoid(logit_e); c_e = fp32(s_e + bias_e), the choice score.  Each of the
 * G groups of E/G consecutive experts scores fp32(c_first + c_second), its two best choice
 * scores; the topk_groups best groups stay eligible; the K best eligible experts by c are
 * chosen, best first (ids[t, k]), and their weights are the renormalised sigmoid scores
 * w_k = s_{ids_k} / S, S the FP32 sum of those scores in slot order, IEEE division.  The
 * routed scaling (2.5) is applied later, by the combine.
 * [vLLM] "MoE und Residual-Stream", bullet "MoE im DeepSeek-V3-Stil" (256 routed experts;
 * sigmoid scores plus a correction bias choose the best 4 of 8 expert groups, then the top 8
 * experts; the renormalised weights are scaled by 2.5) and bullet "FP32-Router"; [SGL]
 * "稠密层与分组 MoE 路由" (grouped top-k from sigmoid scores and the correction bias, FP32
 * coefficients).  The group score as the sum of the two best experts is DeepSeek-V3's rule,
 * which the pages name without restating.  `work` holds 2E + G floats and E + G ints. */
void orc_grouped_topk(int32_t *ids, float *w, const float *logits, const float *bias, int64_t T,
                      int32_t E, int32_t G, int32_t topk_groups, int32_t K, float *work,
                      int32_t *iwork)
{
    float *sc = work, *c = work + E, *gs = work + 2 * E;
    int32_t *allowed = iwork, *gsel = iwork + E;
    int32_t per = E / G;
    for (int64_t t = 0; t < T; ++t) {
        const float *z = logits + t * E;
        for (int32_t e = 0; e < E; ++e) {
            sc[e] = orc_sigmoid_f32(z[e]);
            c[e] = sc[e] + bias[e];
        }
        for (int32_t g = 0; g < G; ++g) {
            int32_t b1 = g * per;
            for (int32_t e = g * per + 1; e < (g + 1) * per; ++e)
                if (ranks_above(c[e], e, c[b1], b1))
                    b1 = e;
            int32_t b2 = -1;
            for (int32_t e = g * per; e < (g + 1) * per; ++e)
                if (e != b1 && (b2 < 0 || ranks_above(c[e], e, c[b2], b2)))
                    b2 = e;
            gs[g] = per > 1 ? c[b1] + c[b2] : c[b1];
            gsel[g] = 0;
        }
        for (int32_t r = 0; r < topk_groups; ++r) {
            int32_t best = -1;
            for (int32_t g = 0; g < G; ++g)
                if (!gsel[g] && (best < 0 || ranks_above(gs[g], g, gs[best], best)))
                    best = g;
            gsel[best] = 1;
        }
        for (int32_t e = 0; e < E; ++e)
            allowed[e] = gsel[e / per];
        float S = 0.0f;
        for (int32_t k = 0; k < K; ++k) {
            int32_t best = -1;
            for (int32_t e = 0; e < E; ++e)
                if (allowed[e] && (best < 0 || ranks_above(c[e], e, c[best], best)))
                    best = e;
            allowed[best] = 0;
            ids[t * K + k] = best;
            S = k == 0 ? sc[best] : S + sc[best];
        }
        for (int32_t k = 0; k < K; ++k)
            w[t * K + k] = sc[ids[t * K + k]] / S;
    }
}

/* ------------------------------------------------------------------------------------------ */
/* KV-cache write (the step the Q/K kernel takes over)                                          */
/* ------------------------------------------------------------------------------------------ */

/* Value of an FP8 E4M3 code (OCP "E4M3FN": 1 sign, 4 exponent bits with bias 7, 3 mantissa
 * bits; exponent field 0 holds the subnormals m * 2^-9; S.1111.111 is NaN; no infinities). */
float orc_fp8_e4m3_to_f32(uint8_t b)
{
    int e = (b >> 3) & 0xf, m = b & 7;
    float mag;
    if (e == 0xf && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexpf((float)m, -9);
    else
        mag = ldexpf(1.0f + (float)m / 8.0f, e - 7);
    return (b & 0x80) ? -mag : mag;
}

/* FP32 -> FP8 E4M3, round to nearest even, saturating: the nearest of the finite codes, ties to
 * the code with an even mantissa; magnitudes from 448 up (infinity included) give +-448; NaN
 * gives 0x7f.  Written as a search over the 127 non-negative finite codes, so that it follows
 * the format's definition directly. */
uint8_t orc_fp8_e4m3_rne(float x)
{
    if (isnan(x))
        return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    float a = fabsf(x);
    if (a >= 448.0f)
        return sign | 0x7e;
    uint8_t lo = 0;                      /* largest code whose value is <= a */
    for (uint8_t c = 1; c <= 0x7e; ++c)
        if (orc_fp8_e4m3_to_f32(c) <= a)
            lo = c;
    uint8_t hi = (uint8_t)(lo + 1);      /* next code up (values grow with the code) */
    float vlo = orc_fp8_e4m3_to_f32(lo), vhi = orc_fp8_e4m3_to_f32(hi);
    double dlo = (double)a - (double)vlo, dhi = (double)vhi - (double)a;  /* exact in double */
    uint8_t pick = dlo < dhi ? lo : (dhi < dlo ? hi : ((lo & 1) ? hi : lo));
    return sign | pick;
}

/* Writes one token's K' rows and V rows into the paged caches, as a separate cache-write kernel
 * would after the Q/K norm: for each token t with slot s = slot_mapping[t] in [0, num_slots),
 *   k_cache[s, h, :] = K'[t, h, :]   and   v_cache[s, h, :] = V[t, h, :]      (h < nk)
 * in BF16 (cache_dtype 0: the bits as they are) or in FP8 E4M3 (cache_dtype 1:
 * fp8(bf16 value / scale), FP32 division, one scale per cache).  Tokens with a negative or
 * out-of-range slot are skipped.  Caches are [num_slots, nk, D] (1 or 2 bytes per element).
 * [vLLM] "MoE und Residual-Stream", change 6 (the Q/K-norm and RoPE kernel also writes K and V
 * into the KV cache); the serving command's FP8 KV cache; [SGL] "目标模型与草稿模型 KV 的统一内存"
 * (KV writes go to the physical slot of each token). */
void orc_kv_cache_write(void *k_cache, void *v_cache, const uint16_t *k, const uint16_t *v,
                        int64_t k_stride, int64_t v_stride, const int64_t *slot_mapping,
                        int64_t T, int32_t nk, int32_t D, int64_t num_slots, int32_t cache_dtype,
                        float k_scale, float v_scale)
{
    for (int64_t t = 0; t < T; ++t) {
        int64_t s = slot_mapping[t];
        if (s < 0 || s >= num_slots)
            continue;
        for (int32_t h = 0; h < nk; ++h)
            for (int32_t d = 0; d < D; ++d) {
                int64_t src_k = t * k_stride + (int64_t)h * D + d;
                int64_t src_v = t * v_stride + (int64_t)h * D + d;
                int64_t dst = (s * nk + h) * (int64_t)D + d;
                if (cache_dtype == 0) {
                    ((uint16_t *)k_cache)[dst] = k[src_k];
                    ((uint16_t *)v_cache)[dst] = v[src_v];
                } else {
                    float kq = orc_bf16_to_f32(k[src_k]) / k_scale;
                    float vq = orc_bf16_to_f32(v[src_v]) / v_scale;
                    ((uint8_t *)k_cache)[dst] = orc_fp8_e4m3_rne(kq);
                    ((uint8_t *)v_cache)[dst] = orc_fp8_e4m3_rne(vq);
                }
            }
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Sigmoid attention-output gate                                                               */
/* ------------------------------------------------------------------------------------------ */

/* out = bf16( attn * sigma ),  sigma = 1 / (1 + e),  e = fp32(exp(-z)),  z = fp32(gate + bias_h).
 * FP32 steps; exp in double rounded to FP32.  bias: [n_heads] FP32.
 * [vLLM] "Attention", bullet "Sigmoid-Output-Gate" (each head's output times sigma(gate + bias),
 * per-head learned bias, a head can be switched off); [SGL] "混合注意力与输出门控" and the
 * kernel-fusion paragraph (bias add, sigmoid and multiply in one kernel). */
void orc_attn_gate(uint16_t *out, const uint16_t *attn, const uint16_t *gate, const float *bias,
                   int64_t T, int32_t nh, int32_t D, int64_t attn_stride, int64_t gate_stride,
                   int64_t out_stride)
{
    for (int64_t t = 0; t < T; ++t) {
        for (int32_t h = 0; h < nh; ++h) {
            for (int32_t d = 0; d < D; ++d) {
                int64_t c = (int64_t)h * D + d;
                float z = orc_bf16_to_f32(gate[t * gate_stride + c]) + bias[h];
                float e = (float)exp(-(double)z);
                float sig = 1.0f / (1.0f + e);
                float a = orc_bf16_to_f32(attn[t * attn_stride + c]);
                out[t * out_stride + c] = orc_bf16_rne(a * sig);
            }
        }
    }
}
