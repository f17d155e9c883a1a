"""Pins of the oracle's grouped top-k routing (CPU only).

Beam routes its 256 experts the way DeepSeek-V3 does ("Serving Reflection Beam auf vLLM ab Tag
0", section "MoE und Residual-Stream", bullets "MoE im DeepSeek-V3-Stil" and "FP32-Router";
"SGLang 支撑编程模型 Beam 生产部署", "稠密层与分组 MoE 路由").  The oracle's exp is pinned against
mpmath at 60 digits; the routing against hand-derived cases (including one where the two-best
group rule excludes the single best expert) and against an independent float64 evaluation on
random logits, wherever the ranking there is not within rounding of a tie.
"""
import math

import mpmath
import numpy as np
import pytest

import oracle

mpmath.mp.dps = 60


def _f32_nearest(v):
    """FP32 rounding (nearest even) of an mpmath value, decided exactly in mpmath."""
    f = np.float32(float(v))
    cands = [np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf))]
    best = min(cands, key=lambda c: (abs(mpmath.mpf(float(c)) - v),
                                     int(np.float32(c).view(np.uint32)) & 1))
    return np.float32(best)


def test_exp_is_the_fp32_rounding_of_the_exact_value():
    g = np.random.default_rng(1)
    xs = np.concatenate([g.uniform(-16.7, 88.7, 3000), g.uniform(-1, 1, 1000),
                         g.normal(0, 3, 1000)]).astype(np.float32)
    for x in xs:
        want = _f32_nearest(mpmath.exp(mpmath.mpf(float(x))))
        assert np.float32(oracle.exp_f32(float(x))) == want, x


def test_sigmoid_values_and_extremes():
    assert oracle.sigmoid_f32(0.0) == 0.5
    assert oracle.sigmoid_f32(100.0) == 1.0
    assert oracle.sigmoid_f32(-100.0) == 0.0           # exp overflows to inf
    sub = oracle.sigmoid_f32(-88.0)                     # 1 / (1 + e^88): a subnormal result
    assert 0.0 < sub < 1.2e-38
    assert sub == pytest.approx(1.0 / (1.0 + math.exp(88.0)), rel=1e-6)
    g = np.random.default_rng(2)
    for z in g.normal(0, 4, 2000).astype(np.float32):
        exact = 1.0 / (1.0 + math.exp(-float(z)))
        got = oracle.sigmoid_f32(float(z))
        # two FP32 roundings (exp, then the add) and the division: within 2 ulps of the value
        assert abs(got - exact) <= 2 * np.spacing(np.float32(exact)), z
        assert oracle.sigmoid_f32(float(z)) + oracle.sigmoid_f32(-float(z)) == \
            pytest.approx(1.0, abs=2e-7)


def test_routing_by_bias_alone():
    # all logits 0: every score is 0.5, so the choice is the bias; bias grows with the index, so
    # groups 4..7 have the best two-expert sums and the best eight experts are 255..248
    z = np.zeros((3, 256), np.float32)
    b = np.arange(256, dtype=np.float32) * np.float32(1e-3)
    ids, w = oracle.grouped_topk(z, b)
    assert (ids == np.arange(255, 247, -1)).all()
    assert (w == 0.125).all()                           # equal scores: 1/8 exactly


def test_group_rule_is_the_sum_of_the_two_best():
    # group 0 holds the single best expert (logit 6) but a weak second (logit -6): its group
    # score 0.9975 + 0.0025 = 1.0 loses to groups 1..7, each with two experts at logit 2
    # (0.8808 + 0.8808); the four best groups are then 1, 2, 3, 4 (equal scores: lower index)
    z = np.full((1, 256), -6.0, np.float32)
    z[0, 0] = 6.0
    for g in range(1, 8):
        z[0, 32 * g + 5] = 2.0
        z[0, 32 * g + 17] = 2.0
    ids, w = oracle.grouped_topk(z, np.zeros(256, np.float32))
    want = [32 * g + o for g in (1, 2, 3, 4) for o in (5, 17)]
    assert ids[0].tolist() == want                       # equal scores: ascending index
    assert 0 not in ids[0]
    # equal scores: equal weights, 1/8 up to the rounding of the FP32 sum of eight equal terms
    assert (w == w[0, 0]).all() and abs(float(w[0, 0]) - 0.125) <= 2 * np.spacing(np.float32(0.125))


def test_ties_go_to_the_lower_index():
    z = np.zeros((2, 256), np.float32)
    ids, _ = oracle.grouped_topk(z, np.zeros(256, np.float32))
    assert (ids == np.arange(8)).all()                  # groups 0..3 tie best; experts 0..7


def test_nan_ranks_below_every_number():
    z = np.zeros((1, 256), np.float32)
    z[0, 3] = np.nan
    b = np.zeros(256, np.float32)
    b[:32] = 1.0                                         # group 0 is the best group
    ids, w = oracle.grouped_topk(z, b)
    assert 3 not in ids[0] and ids[0].tolist() == [0, 1, 2, 4, 5, 6, 7, 8]
    assert np.isfinite(w).all()


def test_random_logits_against_float64_routing():
    g = np.random.default_rng(5)
    T = 400
    z = (g.normal(0, 2, (T, 256))).astype(np.float32)
    b = (g.normal(0, 0.5, 256)).astype(np.float32)
    ids, w = oracle.grouped_topk(z, b)
    checked = 0
    for t in range(T):
        s = 1.0 / (1.0 + np.exp(-z[t].astype(np.float64)))
        c = s + b.astype(np.float64)
        top2 = np.sort(c.reshape(8, 32), axis=1)[:, -2:].sum(axis=1)
        order_g = np.argsort(-top2, kind="stable")
        gsorted = np.sort(top2)[::-1]
        if gsorted[3] - gsorted[4] < 1e-5:
            continue                                     # the group choice is within rounding
        allowed = np.zeros(256, bool)
        for gi in order_g[:4]:
            allowed[32 * gi: 32 * gi + 32] = True
        cc = np.where(allowed, c, -np.inf)
        order_e = np.argsort(-cc, kind="stable")
        csorted = cc[order_e]
        if np.min(csorted[:8] - csorted[1:9]) < 1e-5:
            continue                                     # some rank is within rounding
        assert ids[t].tolist() == order_e[:8].tolist(), t
        ws = s[order_e[:8]] / s[order_e[:8]].sum()
        np.testing.assert_allclose(w[t], ws, rtol=1e-6)
        assert abs(float(np.sum(w[t], dtype=np.float64)) - 1.0) < 1e-6
        assert len({int(i) // 32 for i in ids[t]}) <= 4
        checked += 1
    assert checked > T // 2
