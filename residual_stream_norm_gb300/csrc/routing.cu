// routing.cu -- DeepSeek-V3-style grouped top-k routing (sm_103a).
//
// Pages cited (titles as printed):
//   [vLLM]  "Serving Reflection Beam auf vLLM ab Tag 0"
//   [SGL]   "SGLang 支撑编程模型 Beam 生产部署"
//
// Beam routes 256 experts the way DeepSeek-V3 does: sigmoid scores plus a correction bias pick
// the best 4 of 8 expert groups, then the top 8 experts, whose renormalised scores weight the
// combine ([vLLM] "MoE und Residual-Stream", bullets "MoE im DeepSeek-V3-Stil" and
// "FP32-Router"; [SGL] "稠密层与分组 MoE 路由").  The kernel produces exactly what the MoE
// combine takes: the expert ids per token, best first, and the renormalised FP32 weights
// (the routed scaling is applied by the combine).
//
// One warp per token.  Lane l holds experts 8l..8l+7, so the four lanes of a quad hold one group
// of 32.
// - The ranking decisions are those of the correctly rounded FP32 sigmoids (beam_exp.cuh), the
//   oracle's (see below for how most of them are made on cheaper values).
// - A group's score is the FP32 sum of its two best choice scores.  The quad finds them with two
//   shuffle steps on (key, index) pairs.
// - Every lane ranks the eight group scores.
// - Then eight rounds pick the experts: each lane keeps its eligible experts sorted.  A round
//   takes the warp's best head with two `redux.sync` reductions (the largest key, then the
//   lowest index among the lanes holding it), and the owning lane moves to its next expert.
// The ranking first runs on fast sigmoids (hardware exp) with a proven error bound.  When every
// deciding gap exceeds twice that bound, the decisions are those of the exact scores, and only
// the eight chosen experts need correctly rounded sigmoids, for their weights.  Otherwise, for a
// few tokens in a thousand, all 256 are computed exactly and ranked again.
//
// Ranking order: keys map FP32 values to integers in the same order, so that larger values
// rank higher.  NaN ranks below every number, ineligible experts below NaN, and ties go to the
// lower index.

#include "beam_device.cuh"
#include "beam_exp.cuh"
#include "beam_kernels.h"

namespace beam {
namespace {

constexpr int kExperts = 256;
constexpr int kGroups = 8;
constexpr int kTopkGroups = 4;
constexpr int kTopK = 8;
constexpr int kPerLane = kExperts / 32;  // 8
constexpr int kRouteThreads = 256;      // 8 tokens per CTA pass

// Order-preserving key of an FP32 value: larger values, larger keys; NaN gets 1, below every
// number (the smallest numeric key, that of -inf, is 0x007fffff); 0 marks an ineligible expert.
__device__ __forceinline__ uint32_t rank_key(float v)
{
    const uint32_t u = __float_as_uint(v);
    if (v != v)
        return 1u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_value(uint32_t key)
{
    if (key <= 1u)
        return __uint_as_float(0x7fc00000u);
    return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// (key, index) order: a above b
__device__ __forceinline__ bool above(uint32_t ka, int ia, uint32_t kb, int ib)
{
    return ka > kb || (ka == kb && ia < ib);
}

// Fast FP32 sigmoid for the ranking pass: 1 / (1 + __expf(-z)) with the hardware reciprocal.
// For |z| <= 17 it is within kFastSigmoidErr of the correctly rounded sigmoid.  That bound
// follows from __expf's documented error (2 + 1.173 |x| ulps) through ds = -s (1 - s) de/e, plus
// three FP32 roundings, with room to spare; a sweep of 22.9M arguments measured 1.8e-7.  For
// z > 17 both give exactly 1; for z < -17 both are below 4.2e-8 and closer than 1e-12.
constexpr float kFastSigmoidErr = 1.9073486328125e-06f;  // 2^-19

__device__ __forceinline__ float sigmoid_fast(float z)
{
    const float d = __fadd_rn(1.0f, __expf(-z));
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(d));
    return r;
}

// The routing of one token by one warp, from the lane's 8 scores s (of experts e0..e0+7), its
// biases and logits z.  Lanes k < 8 receive slot k's expert id, score and logit.  With
// `certify`, the scores are within kFastSigmoidErr of the exact ones, and the function returns
// true only if the ranking decisions provably match those the exact scores would give:
// - the 4th and 5th group scores are more than twice their error bound apart;
// - so are every two consecutive chosen experts and the 8th and 9th.
// Sorting is 1-Lipschitz in the max norm, so a gap larger than twice the bound on every score
// leaves the order, the chosen sets and the slot order unchanged.
__device__ __forceinline__ bool route_token(const float (&s)[kPerLane],
                                            const float (&bias)[kPerLane],
                                            const float (&z)[kPerLane], int e0, int lane,
                                            int group, bool certify, int &my_id, float &my_s,
                                            float &my_z)
{
    uint32_t key[kPerLane];
    float cmax = 0.0f;
    bool finite = true;
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        const float c = __fadd_rn(s[i], bias[i]);  // choice score c = s + bias
        key[i] = rank_key(c);
        cmax = fmaxf(cmax, fabsf(c));
        finite = finite && isfinite(c);
    }
    // ---- group score: the FP32 sum of the group's two best choice scores -------------------
    uint32_t k1 = key[0], k2 = 0u;
    int i1 = e0, i2 = 0x7fffffff;
#pragma unroll
    for (int i = 1; i < kPerLane; ++i) {
        if (above(key[i], e0 + i, k1, i1)) {
            k2 = k1, i2 = i1, k1 = key[i], i1 = e0 + i;
        } else if (above(key[i], e0 + i, k2, i2)) {
            k2 = key[i], i2 = e0 + i;
        }
    }
#pragma unroll
    for (int off = 1; off < 4; off <<= 1) {  // merge the two-best lists of the quad
        const uint32_t ok1 = __shfl_xor_sync(0xffffffffu, k1, off);
        const uint32_t ok2 = __shfl_xor_sync(0xffffffffu, k2, off);
        const int oi1 = __shfl_xor_sync(0xffffffffu, i1, off);
        const int oi2 = __shfl_xor_sync(0xffffffffu, i2, off);
        if (above(ok1, oi1, k1, i1)) {  // theirs first: second is the better of ours, their 2nd
            if (above(k1, i1, ok2, oi2))
                k2 = k1, i2 = i1;
            else
                k2 = ok2, i2 = oi2;
            k1 = ok1, i1 = oi1;
        } else if (above(ok1, oi1, k2, i2)) {
            k2 = ok1, i2 = oi1;
        }
    }
    const float gscore = __fadd_rn(key_value(k1), key_value(k2));
    // ---- the topk_groups best groups stay eligible --------------------------------------------
    const uint32_t gkey = rank_key(gscore);
    uint32_t gk[kGroups];
    int rank = 0;
#pragma unroll
    for (int j = 0; j < kGroups; ++j) {
        gk[j] = __shfl_sync(0xffffffffu, gkey, 4 * j);
        rank += above(gk[j], j, gkey, group) ? 1 : 0;
    }
    const bool eligible = rank < kTopkGroups;
    // ---- this lane's eligible experts, best first (odd-even transposition sort) -------------
    uint32_t hk[kPerLane];
    int hi[kPerLane];
    float hs[kPerLane], hz[kPerLane];
#pragma unroll
    for (int i = 0; i < kPerLane; ++i) {
        hk[i] = eligible ? key[i] : 0u;
        hi[i] = e0 + i;
        hs[i] = s[i];
        hz[i] = z[i];
    }
#pragma unroll
    for (int pass = 0; pass < kPerLane; ++pass)
#pragma unroll
        for (int i = pass & 1; i + 1 < kPerLane; i += 2)
            if (above(hk[i + 1], hi[i + 1], hk[i], hi[i])) {
                const uint32_t tk = hk[i];
                const int ti = hi[i];
                const float ts = hs[i], tz = hz[i];
                hk[i] = hk[i + 1], hi[i] = hi[i + 1], hs[i] = hs[i + 1], hz[i] = hz[i + 1];
                hk[i + 1] = tk, hi[i + 1] = ti, hs[i + 1] = ts, hz[i + 1] = tz;
            }
    // ---- the rounds: the warp's best head, then the owner moves on --------------------------
    float cprev = 0.0f, mingap = 3.0e38f;
    const int rounds = certify ? kTopK + 1 : kTopK;  // the ninth only to certify the cut
    for (int k = 0; k < rounds; ++k) {
        const uint32_t best = __reduce_max_sync(0xffffffffu, hk[0]);
        const uint32_t idx =
            __reduce_min_sync(0xffffffffu, hk[0] == best ? (uint32_t)hi[0] : 0xffffffffu);
        const int owner = (int)idx / kPerLane;
        const float sk = __shfl_sync(0xffffffffu, hs[0], owner);
        const float zk = __shfl_sync(0xffffffffu, hz[0], owner);
        const float ck = key_value(best);
        if (k > 0)
            mingap = fminf(mingap, __fsub_rn(cprev, ck));
        cprev = ck;
        if (lane == k) {
            my_s = sk;
            my_z = zk;
            my_id = (int)idx;
        }
        if (lane == owner) {
#pragma unroll
            for (int i = 0; i + 1 < kPerLane; ++i)
                hk[i] = hk[i + 1], hi[i] = hi[i + 1], hs[i] = hs[i + 1], hz[i] = hz[i + 1];
            hk[kPerLane - 1] = 0u;
        }
    }
    if (!certify)
        return true;
    // ---- certificate ---------------------------------------------------------------------------
    // error bounds (generous FP32 arithmetic): a choice score within dc of the exact one, a group
    // score within dg; every |value| <= cm
    const float cm = __int_as_float(__reduce_max_sync(0xffffffffu, __float_as_int(cmax)));
    const bool all_finite = __all_sync(0xffffffffu, finite);
    const float dc = kFastSigmoidErr + cm * 2.384185791015625e-07f;  // + 2 ulp(cm), 2^-22
    const float dg = 2.0f * dc + cm * 4.76837158203125e-07f;          // + 2 ulp(2 cm), 2^-21
    // the 4th and 5th best group scores
    float g4 = 0.0f, g5 = 0.0f;
#pragma unroll
    for (int j = 0; j < kGroups; ++j) {
        int r = 0;
#pragma unroll
        for (int i = 0; i < kGroups; ++i)
            r += above(gk[i], i, gk[j], j) ? 1 : 0;
        if (r == kTopkGroups - 1)
            g4 = key_value(gk[j]);
        if (r == kTopkGroups)
            g5 = key_value(gk[j]);
    }
    return all_finite && cm < 1.0e30f && __fsub_rn(g4, g5) > 2.0f * dg && mingap > 2.0f * dc;
}

// 3 CTAs per SM: more warps to cover the ranking's dependent-instruction latency.  At the 80
// registers this allows the kernel spills a little, and is still faster than at 2 CTAs and 124
// registers without spills (46.4 against 49.4 us at T = 16384; 4 CTAs gave 46.5).
__global__ void __launch_bounds__(kRouteThreads, 3)
    grouped_topk_kernel(const RouteArgs a)
{
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int e0 = lane * kPerLane;
    const int group = lane >> 2;
    pdl_launch_dependents();
    float bias[kPerLane];  // model parameter: read before waiting on the previous kernel
    {
        const float4 b0 = *reinterpret_cast<const float4 *>(a.bias + e0);
        const float4 b1 = *reinterpret_cast<const float4 *>(a.bias + e0 + 4);
        bias[0] = b0.x, bias[1] = b0.y, bias[2] = b0.z, bias[3] = b0.w;
        bias[4] = b1.x, bias[5] = b1.y, bias[6] = b1.z, bias[7] = b1.w;
    }
    pdl_wait();
    const int64_t warps = (int64_t)gridDim.x * (kRouteThreads / 32);
    for (int64_t t = (int64_t)blockIdx.x * (kRouteThreads / 32) + warp; t < a.T; t += warps) {
        const float *zp = a.logits + t * kExperts + e0;
        const float4 z0 = ld_stream_f4(zp), z1 = ld_stream_f4(zp + 4);
        const float z[kPerLane] = {z0.x, z0.y, z0.z, z0.w, z1.x, z1.y, z1.z, z1.w};
        float s[kPerLane];
        int my_id = 0;
        float my_s = 0.0f, my_z = 0.0f;
        // ranking on fast sigmoids; exact ones only for the chosen, unless the ranking is not
        // certified (then every score exactly, and the ranking again)
#pragma unroll
        for (int i = 0; i < kPerLane; ++i)
            s[i] = sigmoid_fast(z[i]);
        if (route_token(s, bias, z, e0, lane, group, true, my_id, my_s, my_z)) {
            my_s = sigmoid_rounded(my_z);
        } else {
#pragma unroll
            for (int i = 0; i < kPerLane; ++i)
                s[i] = sigmoid_rounded(z[i]);
            route_token(s, bias, z, e0, lane, group, false, my_id, my_s, my_z);
        }
        // renormalise: the FP32 sum of the chosen scores in slot order
        float wsum = __shfl_sync(0xffffffffu, my_s, 0);
#pragma unroll
        for (int k = 1; k < kTopK; ++k)
            wsum = __fadd_rn(wsum, __shfl_sync(0xffffffffu, my_s, k));
        if (lane < kTopK) {
            a.ids[t * kTopK + lane] = my_id;
            a.weights[t * kTopK + lane] = __fdiv_rn(my_s, wsum);
        }
    }
}

}  // namespace

cudaError_t launch_grouped_topk(const RouteArgs &a, cudaStream_t stream)
{
    const int64_t ctas = (a.T + kRouteThreads / 32 - 1) / (kRouteThreads / 32);
    const unsigned grid = (unsigned)(ctas < (1 << 20) ? ctas : (1 << 20));
    const cudaError_t e =
        launch_pdl(grouped_topk_kernel, dim3(grid), dim3(kRouteThreads), 0, stream, a);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace beam
