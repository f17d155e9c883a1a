"""Pins of the oracle's boundary chain and MoE combine (CPU only).

The chain (post-RMSNorm -> depth-scaled residual add with BF16-rounded operands -> next
pre-RMSNorm) is defined on "Serving Reflection Beam auf vLLM ab Tag 0" ("MoE und
Residual-Stream": bullets "Sandwich-Norm" and "Tiefenskalierte Residuen"; "Agentengetriebene
Optimierung", changes 1 and 3) and "SGLang 支撑编程模型 Beam 生产部署"
("三明治归一化与深度缩放残差").  Each pin below is checked against something other than the
oracle's own formula: torch's RMSNorm and rounding in double precision, closed forms at special
residual indices, and the unit-variance / unit-RMS invariants the pages state.
"""
import math

import numpy as np
import pytest
import torch

import beam_inputs as bi
import oracle
from tests._util import assert_bf16_close, bf16_ulp_diff, f32_to_bf16_nearest

H = bi.HIDDEN


def f64(u16):
    return oracle.bf16_to_f32(u16).astype(np.float64)


def bf16_ulp(v):
    """Spacing of BF16 numbers at |v| (normal range; 0 maps to the smallest normal spacing)."""
    av = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(av)) - 7)


def lib_rmsnorm(x_u16, w_u16, eps):
    """torch's RMSNorm in float64: x * rsqrt(mean(x^2) + eps) * w."""
    x = torch.from_numpy(f64(x_u16))
    w = torch.from_numpy(f64(w_u16))
    return torch.nn.functional.rms_norm(x, (x.shape[-1],), weight=w, eps=eps).numpy()


def case(T=6, n=5, seed=0, **kw):
    c = bi.boundary_case(T=T, n=n, seed=seed, **kw)
    return {k: (bi.u16(v) if isinstance(v, torch.Tensor) else v) for k, v in c.items()}


def test_n1_post_norm_matches_library_rmsnorm():
    # n = 1: alpha = 0 and s = 1, so h' carries the post-norm output x_hat itself.
    c = case(T=16, seed=1, outlier_frac=0.1, outlier_mult=16.0)
    h_out, y, rstd = oracle.boundary(c["h"], c["x"], c["w_post"], c["w_pre"], n=1)
    want = f32_to_bf16_nearest(lib_rmsnorm(c["x"], c["w_post"], c["eps"]))
    assert_bf16_close(h_out, want, max_ulp=1, min_equal=0.999, what="x_hat vs torch rms_norm")
    xd = f64(c["x"])
    r_exact = 1.0 / np.sqrt(np.mean(xd * xd, axis=1) + c["eps"])
    np.testing.assert_allclose(rstd[:, 0], r_exact, rtol=3e-7)


def test_pre_norm_output_matches_library_rmsnorm():
    c = case(T=16, seed=2)
    h_out, y, rstd = oracle.boundary(c["h"], c["x"], c["w_post"], c["w_pre"], n=7)
    want = f32_to_bf16_nearest(lib_rmsnorm(h_out, c["w_pre"], c["eps"]))
    assert_bf16_close(y, want, max_ulp=1, min_equal=0.999, what="y vs torch rms_norm(h')")
    hd = f64(h_out)
    np.testing.assert_allclose(rstd[:, 1], 1.0 / np.sqrt(np.mean(hd * hd, axis=1) + c["eps"]),
                               rtol=3e-7)


def test_n4_zero_residual_halves_post_norm_output():
    # n = 4: s = sqrt(4) = 2 exactly; with h = 0 the add returns x_hat / 2 with no rounding.
    c = case(T=8, seed=3)
    zero = np.zeros_like(c["h"])
    xhat, _, _ = oracle.boundary(zero, c["x"], c["w_post"], c["w_pre"], n=1)
    h4, _, _ = oracle.boundary(zero, c["x"], c["w_post"], c["w_pre"], n=4)
    assert np.array_equal(oracle.bf16_to_f32(h4), oracle.bf16_to_f32(xhat) * np.float32(0.5))


@pytest.mark.parametrize("n", [4, 16, 64])
def test_square_index_zero_branch_scales_residual(n):
    # x = 0: r = 1/sqrt(eps), x_hat = 0, b = 0, so h' = bf16(alpha * h) with alpha =
    # sqrt((n-1)/n) -- compared against torch rounding of the exact product in double.
    c = case(T=8, seed=4)
    zero = np.zeros_like(c["x"])
    h_out, _, rstd = oracle.boundary(c["h"], zero, c["w_post"], c["w_pre"], n=n)
    want = f32_to_bf16_nearest(f64(c["h"]) * math.sqrt((n - 1) / n))
    d = bf16_ulp_diff(h_out, want)
    assert d.max() <= 1 and np.mean(d == 0) > 0.99
    assert np.allclose(rstd[:, 0], 1.0 / math.sqrt(c["eps"]), rtol=1e-6)


@pytest.mark.parametrize("n", [2, 3, 5, 17, 104, 1_000_000])
def test_depth_scaled_add_within_rounding_bound(n):
    # h' = sqrt((n-1)/n) h + x_hat / sqrt(n) computed exactly in double from the same h and
    # x_hat; three BF16 roundings separate the two (the operands are rounded before the add, so
    # h' is often not the single rounding of the exact sum).
    c = case(T=8, n=n, seed=5)
    xhat, _, _ = oracle.boundary(np.zeros_like(c["h"]), c["x"], c["w_post"], c["w_pre"], n=1)
    h_out, _, _ = oracle.boundary(c["h"], c["x"], c["w_post"], c["w_pre"], n=n)
    a = math.sqrt((n - 1) / n) * f64(c["h"])
    b = f64(xhat) / math.sqrt(n)
    exact = a + b
    got = f64(h_out)
    # each of the three roundings (a, b, a+b) costs at most half a BF16 ulp of its own value;
    # cancellation makes the bound relative to the operands, not to h'
    bound = 0.5 * (bf16_ulp(a) + bf16_ulp(b) + bf16_ulp(got)) * (1 + 2 ** -16)
    assert np.all(np.abs(got - exact) <= bound)


def test_unit_rms_before_weight():
    # With unit weights the pre-norm output has unit RMS up to BF16 rounding.
    c = case(T=32, seed=6, outlier_frac=0.1, outlier_mult=16.0)
    ones = bi.u16(torch.ones(H, dtype=torch.bfloat16))
    h_out, y, _ = oracle.boundary(c["h"], c["x"], ones, ones, n=9)
    ms = np.mean(f64(y) ** 2, axis=1)
    assert np.all(np.abs(ms - 1.0) < 4e-3), ms


def test_constant_row_closed_form():
    # x_j = c for all j: r = 1/sqrt(c^2 + eps) and x_hat_j = bf16(c * r * w_j).
    for cval in (0.5, 2.0, 3.0, 1e-3):
        x = bi.u16(torch.full((1, H), cval, dtype=torch.bfloat16))
        cv = float(oracle.bf16_to_f32(x[0, :1])[0])
        r = 1.0 / math.sqrt(cv * cv + 1e-6)
        ones = bi.u16(torch.ones(H, dtype=torch.bfloat16))
        h_out, _, rstd = oracle.boundary(np.zeros_like(x), x, ones, ones, n=1)
        assert abs(rstd[0, 0] - r) <= 2 ** -23 * r
        assert np.all(h_out == f32_to_bf16_nearest(np.array([cv * r]))[0])


def test_variance_preserved_over_104_adds():
    # The depth-scaled residual keeps unit variance at every depth for unit-variance sublayer
    # outputs ("Tiefenskalierte Residuen"): run the whole batch-1 decode chain (104 boundaries).
    ch = bi.decode_chain()
    h = bi.u16(ch["h0"])
    xs, wpo, wpr = bi.u16(ch["xs"]), bi.u16(ch["w_post"]), bi.u16(ch["w_pre"])
    variances = []
    for i in range(bi.N_BOUNDARIES):
        h, y, _ = oracle.boundary(h, xs[i], wpo[i], wpr[i], n=i + 1)
        variances.append(float(np.var(f64(h))))
        assert np.isfinite(oracle.bf16_to_f32(y)).all()
    v = np.array(variances)
    assert np.all((v > 0.9) & (v < 1.1)), v
    # a chain without depth scaling (plain h + x) would grow to ~104x
    assert v[-1] < 1.1


def test_nonfinite_inputs_propagate():
    c = case(T=3, seed=7)
    x = c["x"].copy()
    x[0, 10] = 0x7FC0  # NaN
    x[1, 20] = 0x7F80  # +inf
    h_out, y, rstd = oracle.boundary(c["h"], x, c["w_post"], c["w_pre"], n=3)
    yf = oracle.bf16_to_f32(y)
    assert np.isnan(yf[0]).all()                 # NaN square -> NaN rstd -> NaN row
    assert rstd[1, 0] == 0.0                     # inf mean square -> r = 0
    assert np.isnan(oracle.bf16_to_f32(h_out)[1, 20])  # inf * 0
    assert np.isfinite(yf[2]).all()              # other tokens untouched


def test_residual_scales_closed_forms():
    assert oracle.residual_scales(1) == (0.0, 1.0)
    a4, s4 = oracle.residual_scales(4)
    assert s4 == 2.0 and a4 == np.float32(math.sqrt(3) / 2)
    for n in (2, 5, 104, 10**6):
        a, s = oracle.residual_scales(n)
        assert a == np.float32(math.sqrt(1 - 1 / n)) and s == np.float32(math.sqrt(n))


# ------------------------------------------------------------------------------------------
# MoE top-K combine
# ------------------------------------------------------------------------------------------

def moe(T=4, K=8, seed=0):
    c = bi.moe_case(T=T, K=K, seed=seed)
    return {k: (bi.u16(v) if (isinstance(v, torch.Tensor) and v.dtype == torch.bfloat16)
                else (v.numpy() if isinstance(v, torch.Tensor) else v)) for k, v in c.items()}


def test_one_hot_weights_give_scaled_expert():
    c = moe(T=8, seed=1)
    T, K = c["topk_w"].shape
    for pick in (0, 3, 7):
        w = np.zeros((T, K), dtype=np.float32)
        w[:, pick] = 1.0
        *_, x = oracle.moe_combine_boundary(c["h"], c["e"], w, c["w_post"], c["w_pre"], n=8,
                                            return_x=True)
        want = f32_to_bf16_nearest(2.5 * f64(c["e"][:, pick, :]))
        assert np.array_equal(x, want)


def test_uniform_weights_identical_experts_exact():
    # c_k = 2.5 / 8 = 0.3125 exactly and every partial sum is exact: x = bf16(2.5 e).
    c = moe(T=4, seed=2)
    e1 = c["e"][:, :1, :]
    e = np.repeat(e1, 8, axis=1)
    w = np.full((4, 8), 0.125, dtype=np.float32)
    *_, x = oracle.moe_combine_boundary(c["h"], e, w, c["w_post"], c["w_pre"], n=8,
                                        return_x=True)
    assert np.array_equal(x, f32_to_bf16_nearest(2.5 * f64(e1[:, 0, :])))


def test_combine_matches_exact_weighted_sum():
    c = moe(T=16, seed=3)
    *_, x = oracle.moe_combine_boundary(c["h"], c["e"], c["topk_w"], c["w_post"], c["w_pre"],
                                        n=8, return_x=True)
    cw = (c["topk_w"].astype(np.float32) * np.float32(2.5)).astype(np.float64)
    exact = np.einsum("tk,tkh->th", cw, f64(c["e"]))
    d = bf16_ulp_diff(x, f32_to_bf16_nearest(exact))
    assert d.max() <= 1 and np.mean(d == 0) > 0.999


def test_combine_then_boundary_is_the_boundary_chain():
    c = moe(T=8, seed=4)
    h1, y1, r1, x = oracle.moe_combine_boundary(c["h"], c["e"], c["topk_w"], c["w_post"],
                                                c["w_pre"], n=10, return_x=True)
    h2, y2, r2 = oracle.boundary(c["h"], x, c["w_post"], c["w_pre"], n=10)
    assert np.array_equal(h1, h2) and np.array_equal(y1, y2) and np.array_equal(r1, r2)


# ------------------------------------------------------------------------------------------
# the exact row sum (the sum of squares is taken exactly and rounded once to FP32)
# ------------------------------------------------------------------------------------------

def _nearest_f32(fr):
    """FP32 nearest to a non-negative Fraction, ties to even (exact selection by comparison)."""
    from fractions import Fraction
    c = np.float32(float(fr))
    cands = {c, np.nextafter(c, np.float32(np.inf)), np.nextafter(c, np.float32(0))}
    best = None
    for v in sorted(cands):
        d = abs(Fraction(float(v)) - fr)
        key = (d, int(np.array(v, np.float32).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, v)
    return best[1]


def test_exact_sum_matches_rational_arithmetic():
    from fractions import Fraction
    g = np.random.Generator(np.random.PCG64(3))
    cases = [
        [1.0, 2.0 ** -24],                       # exact tie: stays on the even neighbour
        [1.0, 2.0 ** -24, 2.0 ** -60],           # just above the tie: up (double sum misses it)
        [1.0, 2.0 ** -24, 2.0 ** -149],          # above the tie by one subnormal
        [1.0 + 2.0 ** -23, 2.0 ** -24],          # tie, odd neighbour: up
        [2.0 ** -149] * 7,                       # subnormal sum
        [3.0e38, 3.0e38],                        # overflow to inf
        [],
        list(g.standard_normal(5120).astype(np.float32) ** 2),
        list((g.standard_normal(4096) * 2.0 ** g.integers(-60, 60, 4096)).astype(np.float32) ** 2),
    ]
    for terms in cases:
        t = np.array(terms, dtype=np.float32)
        got = oracle.exact_sum_f32(t)
        exact = sum((Fraction(float(v)) for v in t), Fraction(0))
        want = np.float32(np.inf) if exact > Fraction(float(np.finfo(np.float32).max)) * \
            (1 + Fraction(1, 2 ** 25)) else _nearest_f32(exact)
        assert np.float32(got) == want, (terms[:4], got, want)
    assert np.isnan(oracle.exact_sum_f32(np.array([1.0, np.nan], np.float32)))
    assert oracle.exact_sum_f32(np.array([1.0, np.inf], np.float32)) == np.inf


def test_near_tie_row_sum_rounds_up():
    # squares 1, 2^-24, 2^-60 of BF16 values 1, 2^-12, 2^-30: the exact sum lies just above the
    # midpoint between 1 and 1 + 2^-23, so its FP32 rounding is 1 + 2^-23.
    H = 8
    x = np.zeros((1, H), np.float32)
    x[0, :3] = [1.0, 2.0 ** -12, 2.0 ** -30]
    xb = oracle.bf16_rne(x)
    ones = oracle.bf16_rne(np.ones(H, np.float32))
    _, _, rstd = oracle.boundary(np.zeros_like(xb), xb, ones, ones, n=1, eps=0.0)
    ms = np.float32(1.0 + 2.0 ** -23)
    assert rstd[0, 0] == np.float32(1.0) / np.sqrt(ms / np.float32(H))
