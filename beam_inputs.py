"""Seeded synthetic inputs for the Beam sublayer-boundary path.

Shared by the tests, the smoke check and the benchmark, for both the CUDA library and the CPU
oracle.  This module holds none of the method's arithmetic: only random draws (numpy PCG64,
seeded) and the FP32 -> BF16 storage conversion of torch on the CPU.

BF16 tensors are returned as CPU ``torch.bfloat16`` tensors; ``u16(t)`` gives the numpy
``uint16`` bit patterns the oracle takes.

Shapes follow the Beam decoder the pages describe: hidden 5120, 48 query / 8 KV heads of
dimension 128, top-8 of 256 experts, 104 sublayer boundaries (52 layers x 2).
"""
from __future__ import annotations

import numpy as np
import torch

HIDDEN = 5120
N_Q_HEADS = 48
N_KV_HEADS = 8
HEAD_DIM = 128
TOP_K = 8
N_BOUNDARIES = 104
ROUTED_SCALING = 2.5
EPS = 1e-6
ROPE_THETA = 10000.0
SSMAX_BASE = 2048.0
SSMAX_EXP = 0.1
MAX_POS = 1 << 20  # 1M-token context


def rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def to_bf16(a: np.ndarray) -> torch.Tensor:
    """FP32 numpy array -> CPU bf16 tensor (torch's round-to-nearest-even conversion)."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)


def u16(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def from_u16(a: np.ndarray) -> torch.Tensor:
    """numpy uint16 bit patterns -> CPU bf16 tensor."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).view(
        torch.bfloat16)


def normal(g: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    out = g.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        out *= np.float32(std)
    return out


def norm_weight(g: np.random.Generator, n: int) -> torch.Tensor:
    """RMSNorm weight 1 + 0.1 * N(0, 1), drawn in FP32 and stored as BF16."""
    return to_bf16(1.0 + 0.1 * normal(g, (n,)))


def token_scaled(g: np.random.Generator, T: int, H: int, lo: float = 0.5, hi: float = 4.0,
                 outlier_frac: float = 0.0, outlier_mult: float = 1.0,
                 scales: np.ndarray | None = None) -> torch.Tensor:
    """Rows N(0, 1) * s_t with a per-token scale s_t ~ U(lo, hi); a fraction of the tokens
    (at least one when the fraction is positive and T > 0) is multiplied by ``outlier_mult``."""
    if scales is None:
        scales = g.uniform(lo, hi, size=T).astype(np.float32)
    a = normal(g, (T, H))
    a *= scales[:, None]
    if outlier_frac > 0 and T > 0:
        n_out = max(1, int(round(outlier_frac * T)))
        idx = g.choice(T, size=n_out, replace=False)
        a[idx] *= np.float32(outlier_mult)
    return to_bf16(a)


# ---------------------------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------------------------

def boundary_case(T: int = 4, H: int = HIDDEN, n: int = 5, seed: int = 0,
                  outlier_frac: float = 0.0, outlier_mult: float = 1.0,
                  shared_scale: bool = True) -> dict:
    """Single boundary: h, x ~ N(0,1) * s_t with s_t ~ U(0.5, 4) per token; norm weights
    1 + 0.1 N(0,1).  ``shared_scale`` uses one s_t per token for both h and x."""
    g = rng(seed)
    s_t = g.uniform(0.5, 4.0, size=T).astype(np.float32)
    h = token_scaled(g, T, H, scales=s_t)
    x = token_scaled(g, T, H, scales=s_t if shared_scale else None,
                     outlier_frac=outlier_frac, outlier_mult=outlier_mult)
    return dict(h=h, x=x, w_post=norm_weight(g, H), w_pre=norm_weight(g, H), n=n, eps=EPS)


def decode_chain(H: int = HIDDEN, steps: int = N_BOUNDARIES, seed: int = 0,
                 outlier_frac: float = 0.05, outlier_mult: float = 8.0) -> dict:
    """Batch-1 decode over ``steps`` boundaries n = 1..steps: h0 ~ N(0,1); a fresh sublayer
    output x_n ~ N(0,1) per boundary, of which a fraction (over the chain's draws) is scaled
    by ``outlier_mult``; own post/pre norm weights per boundary."""
    g = rng(seed)
    h0 = to_bf16(normal(g, (1, H)))
    xs = normal(g, (steps, 1, H))
    n_out = max(1, int(round(outlier_frac * steps)))
    idx = g.choice(steps, size=n_out, replace=False)
    xs[idx] *= np.float32(outlier_mult)
    w_post = torch.stack([norm_weight(g, H) for _ in range(steps)])
    w_pre = torch.stack([norm_weight(g, H) for _ in range(steps)])
    return dict(h0=h0, xs=to_bf16(xs), w_post=w_post, w_pre=w_pre, outliers=np.sort(idx),
                eps=EPS)


def topk_weights(g: np.random.Generator, T: int, K: int = TOP_K) -> np.ndarray:
    """Renormalised FP32 routing weights of the K selected experts: sigmoid-like scores
    s ~ U(0, 1), w_k = s_k / sum_j s_j in FP32 (the router's renormalisation; done by the
    caller, not by the combine)."""
    s = g.uniform(0.0, 1.0, size=(T, K)).astype(np.float32)
    s = np.maximum(s, np.float32(1e-6))
    return (s / s.sum(axis=1, dtype=np.float32, keepdims=True)).astype(np.float32)


def moe_case(T: int = 128, H: int = HIDDEN, K: int = TOP_K, layer: int = 3, seed: int = 0,
             expert_std: float = 1.0) -> dict:
    """MoE boundary: top-K expert outputs e [T, K, H] ~ N(0, 1); FP32 renormalised weights;
    residual h ~ N(0, 1); residual index n = 2 * layer + 2."""
    g = rng(seed)
    h = to_bf16(normal(g, (T, H)))
    e = to_bf16(normal(g, (T, K, H), std=expert_std))
    w = torch.from_numpy(topk_weights(g, T, K))
    return dict(h=h, e=e, topk_w=w, w_post=norm_weight(g, H), w_pre=norm_weight(g, H),
                n=2 * layer + 2, eps=EPS, routed_scaling=ROUTED_SCALING)


def attn_qk_case(T: int, n_q: int = N_Q_HEADS, n_kv: int = N_KV_HEADS, D: int = HEAD_DIM,
                 seed: int = 0, pos_mode: str = "uniform", pos_start: int = 98_304) -> dict:
    """Q [T, n_q, D], K [T, n_kv, D] ~ N(0, 1); per-head norm weights 1 + 0.1 N(0,1) of length
    D (one for Q, one for K); 0-based positions either U[0, 2^20) ("uniform") or a contiguous
    run starting at ``pos_start`` ("contiguous", a prefill chunk at ~100K context)."""
    g = rng(seed)
    q = to_bf16(normal(g, (T, n_q, D)))
    k = to_bf16(normal(g, (T, n_kv, D)))
    wq, wk = norm_weight(g, D), norm_weight(g, D)
    if pos_mode == "uniform":
        pos = g.integers(0, MAX_POS, size=T, dtype=np.int64)
    elif pos_mode == "contiguous":
        pos = pos_start + np.arange(T, dtype=np.int64)
    else:
        raise ValueError(pos_mode)
    return dict(q=q, k=k, wq=wq, wk=wk, pos=torch.from_numpy(pos), eps=EPS)


def kv_cache_case(T: int, n_kv: int = N_KV_HEADS, D: int = HEAD_DIM, slots_per_token: int = 4,
                  pad_frac: float = 0.05, oob_frac: float = 0.02, seed: int = 0) -> dict:
    """V [T, n_kv, D] ~ N(0, 1) and a slot mapping into a paged cache of
    ``num_slots = slots_per_token * T`` slots: each token gets a distinct random slot, except a
    ``pad_frac`` share of padding tokens (slot -1) and an ``oob_frac`` share mapped past the end
    of the cache (which must not be written)."""
    g = rng(seed)
    v = to_bf16(normal(g, (T, n_kv, D)))
    num_slots = slots_per_token * T
    slots = g.permutation(num_slots)[:T].astype(np.int64)
    u = g.random(T)
    slots[u < pad_frac] = -1
    slots[(u >= pad_frac) & (u < pad_frac + oob_frac)] = num_slots + g.integers(0, 1000)
    return dict(v=v, slot_mapping=torch.from_numpy(slots), num_slots=num_slots)


N_EXPERTS = 256
N_GROUPS = 8
TOPK_GROUPS = 4


def routing_case(T: int, seed: int = 0, logit_std: float = 1.5, bias_std: float = 0.3) -> dict:
    """FP32 router logits [T, 256] ~ N(0, logit_std^2) and an FP32 correction bias [256] ~
    N(0, bias_std^2): the inputs of the grouped routing."""
    g = rng(seed)
    logits = torch.from_numpy(normal(g, (T, N_EXPERTS), std=logit_std))
    bias = torch.from_numpy(normal(g, (N_EXPERTS,), std=bias_std))
    return dict(logits=logits, bias=bias)


def gate_case(T: int, n_heads: int = N_Q_HEADS, D: int = HEAD_DIM, seed: int = 0) -> dict:
    """attn ~ N(0, 1); gate ~ N(0, 2) read as variance 2 (std sqrt 2); per-head bias ~ N(0, 1)
    in FP32."""
    g = rng(seed)
    attn = to_bf16(normal(g, (T, n_heads * D)))
    gate = to_bf16(normal(g, (T, n_heads * D), std=float(np.sqrt(2.0))))
    bias = torch.from_numpy(normal(g, (n_heads,)))
    return dict(attn=attn, gate=gate, bias=bias)


def prefill_boundary_case(T: int = 16384, H: int = HIDDEN, seed: int = 0) -> dict:
    """8 x 2048 prefill: x = N(0,1) * s_t, s_t ~ U(0.5, 4), 1 % of tokens x16; h ~ N(0, 1);
    one weight pair per residual index n = 1..104 (the launch for n uses pair n-1)."""
    g = rng(seed)
    h = to_bf16(normal(g, (T, H)))
    x = token_scaled(g, T, H, outlier_frac=0.01, outlier_mult=16.0)
    w_post = torch.stack([norm_weight(g, H) for _ in range(N_BOUNDARIES)])
    w_pre = torch.stack([norm_weight(g, H) for _ in range(N_BOUNDARIES)])
    return dict(h=h, x=x, w_post=w_post, w_pre=w_pre, eps=EPS)


TP_RANKS = 8


def allreduce_case(T: int = 128, H: int = HIDDEN, P: int = TP_RANKS, n: int = 7, seed: int = 0,
                   outlier_frac: float = 0.01, outlier_mult: float = 16.0) -> dict:
    """Tensor-parallel sublayer output over P ranks: partials x_p [P, T, H], each
    N(0, 1) * s_t / sqrt(P) with one s_t ~ U(0.5, 4) per token shared by the ranks (so the sum
    has the prefill case's spread), a fraction of the tokens x``outlier_mult`` on every rank;
    h ~ N(0, 1); norm weights 1 + 0.1 N(0, 1); residual index n."""
    g = rng(seed)
    s_t = g.uniform(0.5, 4.0, size=T).astype(np.float32) / np.float32(np.sqrt(P))
    if outlier_frac > 0 and T > 0:
        idx = g.choice(T, size=max(1, int(round(outlier_frac * T))), replace=False)
        s_t[idx] *= np.float32(outlier_mult)
    parts = normal(g, (P, T, H))
    parts *= s_t[None, :, None]
    h = to_bf16(normal(g, (T, H)))
    return dict(h=h, parts=to_bf16(parts), w_post=norm_weight(g, H), w_pre=norm_weight(g, H),
                n=n, eps=EPS)
