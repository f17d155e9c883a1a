"""Pins of the oracle's attention-side operations (CPU only).

Per-head Q/K RMSNorm fused with RoPE (sliding-window layers) or the SSMax query scale (NoPE
layers), and the sigmoid output gate: "Serving Reflection Beam auf vLLM ab Tag 0", section
"Attention" (bullets "Hybride Sliding-Window- und NoPE-Schichten", "SSMax auf NoPE-Schichten",
"GQA mit Per-Head-Q/K-Norm", "Sigmoid-Output-Gate"), and "SGLang 支撑编程模型 Beam 生产部署"
("混合注意力与输出门控"; the SSMax paragraph under "稠密层与分组 MoE 路由").  Each pin checks
the oracle against a closed form or against torch in double precision.
"""
import math

import numpy as np
import pytest
import torch

import beam_inputs as bi
import oracle
from tests._util import assert_bf16_close, bf16_ulp_diff, f32_to_bf16_nearest

D = bi.HEAD_DIM


def f64(u16):
    return oracle.bf16_to_f32(u16).astype(np.float64)


def qk(T=4, seed=0, n_q=bi.N_Q_HEADS, n_kv=bi.N_KV_HEADS, pos_mode="uniform"):
    c = bi.attn_qk_case(T=T, n_q=n_q, n_kv=n_kv, seed=seed, pos_mode=pos_mode)
    return {k: (bi.u16(v) if (isinstance(v, torch.Tensor) and v.dtype == torch.bfloat16)
                else (v.numpy() if isinstance(v, torch.Tensor) else v)) for k, v in c.items()}


def lib_head_norm(x_u16, w_u16, eps):
    x = torch.from_numpy(f64(x_u16))
    w = torch.from_numpy(f64(w_u16))
    return torch.nn.functional.rms_norm(x, (x.shape[-1],), weight=w, eps=eps).numpy()


# ------------------------------------------------------------------------------------------
# RoPE
# ------------------------------------------------------------------------------------------

def test_rope_at_position_zero_is_plain_head_norm():
    c = qk(T=3, seed=1)
    pos = np.zeros(3, dtype=np.int64)
    q, k = oracle.qk_norm_rope(c["q"], c["k"], c["wq"], c["wk"], pos)
    assert_bf16_close(q, f32_to_bf16_nearest(lib_head_norm(c["q"], c["wq"], c["eps"])),
                      what="q at pos 0")
    assert_bf16_close(k, f32_to_bf16_nearest(lib_head_norm(c["k"], c["wk"], c["eps"])),
                      what="k at pos 0")


@pytest.mark.parametrize("theta", [10000.0, 500000.0, 1.0])
def test_rope_is_complex_rotation_of_normalised_pairs(theta):
    # Half-rotation convention: element i pairs with i + D/2 as the complex number
    # qhat_i + 1j * qhat_{i+D/2}, multiplied by exp(1j * angle_i).  The angle is the FP32 product
    # fp32(pos) * fp32(theta^(-2i/D)), formed here with numpy float32.
    c = qk(T=5, seed=2)
    pos = c["pos"]
    q, k = oracle.qk_norm_rope(c["q"], c["k"], c["wq"], c["wk"], pos, theta=theta)
    i = np.arange(D // 2)
    inv_freq = (np.float64(theta) ** (-2.0 * i / D)).astype(np.float32)
    ang = (pos.astype(np.float32)[:, None] * inv_freq[None, :]).astype(np.float64)
    rot = np.exp(1j * ang)[:, None, :]
    for got, src, w in ((q, c["q"], c["wq"]), (k, c["k"], c["wk"])):
        xh = lib_head_norm(src, w, c["eps"])
        z = (xh[..., : D // 2] + 1j * xh[..., D // 2:]) * rot
        want = np.concatenate([z.real, z.imag], axis=-1)
        assert_bf16_close(got, f32_to_bf16_nearest(want), max_ulp=1, min_equal=0.995,
                          what=f"rope theta={theta}")


def test_rope_preserves_pair_norms():
    c = qk(T=4, seed=3)
    q, _ = oracle.qk_norm_rope(c["q"], c["k"], c["wq"], c["wk"], c["pos"])
    q0, _ = oracle.qk_norm_rope(c["q"], c["k"], c["wq"], c["wk"], np.zeros(4, np.int64))
    a, b = f64(q), f64(q0)
    na = a[..., : D // 2] ** 2 + a[..., D // 2:] ** 2
    nb = b[..., : D // 2] ** 2 + b[..., D // 2:] ** 2
    np.testing.assert_allclose(na, nb, rtol=2 ** -6, atol=1e-6)


def test_rope_inv_freq_closed_form():
    f = oracle.rope_inv_freq(10000.0, D)
    assert f[0] == 1.0
    assert f[32] == np.float32(0.01)           # theta^(-1/2) = 1/100
    assert f[48] == np.float32(0.001)          # theta^(-3/4)


# ------------------------------------------------------------------------------------------
# SSMax
# ------------------------------------------------------------------------------------------

def test_ssmax_first_position():
    # 1-based p = 1 (0-based pos 0): (1 + 1/2048)^0.1 = exp(0.1 * log1p(1/2048)).
    s = oracle.ssmax_scale(0)
    assert s == np.float32(math.exp(0.1 * math.log1p(1 / 2048)))
    # first-order expansion 1 + 0.1/2048, to within one FP32 ulp at 1 (the value is FP32)
    assert abs(s - (1 + 0.1 / 2048)) <= 2 ** -23


def test_ssmax_one_and_zero_based_forms_agree_with_powers_of_two():
    # 1 + p/2048 = 32 gives 32^0.1 = sqrt(2); 1 + p/2048 = 1024 gives exactly 2.
    p_sqrt2 = 31 * 2048            # 1-based
    p_two = 1023 * 2048
    assert oracle.ssmax_scale(p_sqrt2 - 1) == np.float32(math.sqrt(2))
    assert oracle.ssmax_scale(p_two - 1) == 2.0
    # monotone in position and > 1
    vals = [oracle.ssmax_scale(p) for p in (0, 10, 511, 4096, 100_000, (1 << 20) - 1)]
    assert all(v > 1.0 for v in vals) and all(a < b for a, b in zip(vals, vals[1:]))


def test_ssmax_scales_queries_only_after_norm():
    c = qk(T=2, seed=4)
    pos = np.array([1023 * 2048 - 1, 0], dtype=np.int64)   # scale 2 exactly, then ~1
    q, k = oracle.qk_norm_ssmax(c["q"], c["k"], c["wq"], c["wk"], pos)
    plain_q = f32_to_bf16_nearest(lib_head_norm(c["q"], c["wq"], c["eps"]))
    plain_k = f32_to_bf16_nearest(lib_head_norm(c["k"], c["wk"], c["eps"]))
    # token 0: a power-of-two scale commutes with the rounding
    assert_bf16_close(oracle.bf16_rne(oracle.bf16_to_f32(q[0]) * np.float32(0.5)), plain_q[0],
                      what="q/2 at scale 2")
    # keys never see the scale
    assert_bf16_close(k, plain_k, what="k unscaled")
    assert np.array_equal(k, oracle.qk_norm_ssmax(c["q"], c["k"], c["wq"], c["wk"],
                                                  np.array([5, 77], np.int64))[1])


# ------------------------------------------------------------------------------------------
# sigmoid output gate
# ------------------------------------------------------------------------------------------

def gate(T=4, seed=0):
    c = bi.gate_case(T=T, seed=seed)
    return bi.u16(c["attn"]), bi.u16(c["gate"]), c["bias"].numpy()


def test_gate_bias_minus_inf_switches_head_off():
    attn, g, bias = gate(seed=1)
    bias = bias.copy()
    bias[5] = -np.inf
    out = oracle.attn_gate(attn, g, bias, bi.N_Q_HEADS, D)
    head = oracle.bf16_to_f32(out).reshape(4, bi.N_Q_HEADS, D)[:, 5]
    assert np.all(head == 0.0)
    others = oracle.bf16_to_f32(out).reshape(4, bi.N_Q_HEADS, D)[:, 6]
    assert np.any(others != 0.0)


def test_gate_bias_plus_inf_passes_attention_through():
    attn, g, _ = gate(seed=2)
    bias = np.full(bi.N_Q_HEADS, np.inf, dtype=np.float32)
    assert np.array_equal(oracle.attn_gate(attn, g, bias, bi.N_Q_HEADS, D), attn)


def test_gate_zero_logit_halves():
    attn, g, _ = gate(seed=3)
    zero = np.zeros_like(g)
    out = oracle.attn_gate(attn, zero, np.zeros(bi.N_Q_HEADS, np.float32), bi.N_Q_HEADS, D)
    assert np.array_equal(oracle.bf16_to_f32(out), oracle.bf16_to_f32(attn) * np.float32(0.5))


def test_gate_matches_library_sigmoid():
    attn, g, bias = gate(T=16, seed=4)
    z = torch.from_numpy(f64(g).reshape(16, bi.N_Q_HEADS, D) + bias.astype(np.float64)[:, None])
    want = f64(attn) * torch.sigmoid(z).numpy().reshape(16, -1)
    out = oracle.attn_gate(attn, g, bias, bi.N_Q_HEADS, D)
    assert_bf16_close(out, f32_to_bf16_nearest(want), what="gate vs torch.sigmoid")
    d = bf16_ulp_diff(out, f32_to_bf16_nearest(want))
    assert d.max() <= 1
