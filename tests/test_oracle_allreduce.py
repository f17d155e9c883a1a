"""Pins of the oracle's tensor-parallel all-reduce boundary (CPU only).

Under tensor parallelism each rank holds a partial sublayer output; "Serving Reflection Beam auf
vLLM ab Tag 0" ("Agentengetriebene Optimierung", change 3) runs both TP all-reduces of a layer
inside the norm kernel, and "SGLang 支撑编程模型 Beam 生产部署" (kernel-fusion paragraph) fuses the
all-reduce with the output norm, the scaled residual add and the next input norm.  The reading
pinned here: the BF16 partials are summed in rank order in FP32, starting from rank 0's value,
and the sum is rounded once to BF16 before the boundary chain.

Each pin checks the oracle against something other than its own loop: the plain boundary
(P = 1 and exact splits), numpy's IEEE FP32 additions with torch's BF16 rounding, a constructed
case whose result depends on the rank order, exact rational arithmetic for the error bound, and
signed zeros.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import beam_inputs as bi
import oracle
from tests._util import f32_to_bf16_nearest

H = bi.HIDDEN


def case(T=6, P=8, n=7, seed=0, H=H):
    c = bi.allreduce_case(T=T, H=H, P=P, n=n, seed=seed)
    return {k: (bi.u16(v) if isinstance(v, torch.Tensor) else v) for k, v in c.items()}


def same(a, b, what):
    for x, y, name in zip(a, b, ("h'", "y", "rstd")):
        x, y = np.asarray(x), np.asarray(y)
        assert np.array_equal(x.view(np.uint32) if x.dtype == np.float32 else x,
                              y.view(np.uint32) if y.dtype == np.float32 else y), f"{what} {name}"


def test_single_rank_is_the_plain_boundary():
    c = case(P=1, seed=1)
    got = oracle.allreduce_boundary(c["h"], c["parts"], c["w_post"], c["w_pre"], c["n"])
    want = oracle.boundary(c["h"], c["parts"][0], c["w_post"], c["w_pre"], c["n"])
    same(got, want, "P=1")


@pytest.mark.parametrize("P", [2, 4, 8])
def test_exact_split_gives_the_boundary_of_the_whole(P):
    # x / P is exact in BF16 for normal x and a power-of-two P, and every partial sum
    # (p + 1) x / P needs at most 8 + 3 significant bits: the FP32 sum is x exactly.
    c = case(T=5, P=1, seed=2)
    x = oracle.bf16_to_f32(c["parts"][0])
    assert np.all(np.abs(x[x != 0]) > 2.0 ** -100)
    part = oracle.bf16_rne(x / np.float32(P))
    assert np.array_equal(oracle.bf16_to_f32(part) * np.float32(P), x)
    parts = np.stack([part] * P)
    got = oracle.allreduce_boundary(c["h"], parts, c["w_post"], c["w_pre"], 9, return_x=True)
    want = oracle.boundary(c["h"], c["parts"][0], c["w_post"], c["w_pre"], 9)
    assert np.array_equal(got[3], c["parts"][0])
    same(got[:3], want, f"P={P} exact split")


def test_rank_permutation_changes_nothing_when_every_partial_sum_is_exact():
    # small integers times a common power of two: every FP32 partial sum is exact, so any rank
    # order gives the same x and the same outputs
    g = bi.rng(3)
    P, T = 8, 4
    ints = g.integers(-60, 61, size=(P, T, H)).astype(np.float32)
    parts = oracle.bf16_rne(ints * np.float32(2.0 ** -5))
    c = case(T=T, P=P, seed=3)
    ref = oracle.allreduce_boundary(c["h"], parts, c["w_post"], c["w_pre"], 5, return_x=True)
    for perm in (np.arange(P)[::-1], g.permutation(P)):
        got = oracle.allreduce_boundary(c["h"], parts[perm].copy(), c["w_post"], c["w_pre"], 5,
                                        return_x=True)
        assert np.array_equal(got[3], ref[3])
        same(got[:3], ref[:3], f"perm {perm}")


def test_rank_order_decides_where_the_fp32_sum_rounds():
    # partials (1, 2^-8, 2^-24, 2^-24): in rank order each 2^-24 is half an FP32 ulp of the
    # running sum and rounds away (ties to even), leaving 1 + 2^-8, a BF16 tie that rounds to 1;
    # in reverse order the small terms add up first and the sum 1 + 2^-8 + 2^-23 rounds up to
    # the next BF16 value 1 + 2^-7.  The exact sum (and a double accumulation) gives the latter
    # in both orders, so this separates FP32 rank-order accumulation from exact summation.
    vals = np.array([1.0, 2.0 ** -8, 2.0 ** -24, 2.0 ** -24], np.float32)
    T, P = 1, 4
    c = case(T=T, P=P, seed=4)
    fwd = np.stack([oracle.bf16_rne(np.full((T, H), v, np.float32)) for v in vals])
    x_fwd = oracle.allreduce_boundary(c["h"], fwd, c["w_post"], c["w_pre"], 3, return_x=True)[3]
    x_rev = oracle.allreduce_boundary(c["h"], fwd[::-1].copy(), c["w_post"], c["w_pre"], 3,
                                      return_x=True)[3]
    assert np.all(oracle.bf16_to_f32(x_fwd) == 1.0)
    assert np.all(oracle.bf16_to_f32(x_rev) == np.float32(1.0 + 2.0 ** -7))


def test_reduced_x_matches_numpy_fp32_adds_and_torch_rounding():
    # numpy's float32 addition is IEEE round-to-nearest-even and torch converts to BF16 with
    # RNE: an implementation of the same reading that shares nothing with the C oracle.
    for P, seed in ((2, 5), (3, 6), (8, 7)):
        c = case(T=9, P=P, seed=seed)
        f = oracle.bf16_to_f32(c["parts"])
        acc = f[0].copy()
        for p in range(1, P):
            acc = (acc + f[p]).astype(np.float32)
        want_x = f32_to_bf16_nearest(acc)
        got = oracle.allreduce_boundary(c["h"], c["parts"], c["w_post"], c["w_pre"], c["n"],
                                        return_x=True)
        assert np.array_equal(got[3], want_x)
        # and the chain after it is the plain boundary of that x
        same(got[:3], oracle.boundary(c["h"], want_x, c["w_post"], c["w_pre"], c["n"]),
             f"P={P} chain")


def test_reduced_x_within_the_rank_order_error_bound():
    # |x - sum_p x_p| <= (P - 1) u sum_p |x_p| + ulp_bf16(x) / 2 with u = 2^-24: each FP32 add
    # errs by at most u times its result, which is at most the sum of magnitudes so far.  A
    # dropped, doubled or sign-flipped partial breaks it by orders of magnitude.
    P = 8
    c = case(T=3, P=P, seed=8, H=64)
    got_x = oracle.allreduce_boundary(c["h"], c["parts"], c["w_post"], c["w_pre"], 5,
                                      return_x=True)[3]
    f = oracle.bf16_to_f32(c["parts"]).astype(np.float64)
    xv = oracle.bf16_to_f32(got_x).astype(np.float64)
    for t in range(3):
        for j in range(64):
            exact = sum(Fraction(float(f[p, t, j])) for p in range(P))
            mag = sum(abs(Fraction(float(f[p, t, j]))) for p in range(P))
            ax = abs(xv[t, j])
            half_ulp = Fraction(2) ** (int(np.floor(np.log2(ax))) - 8) if ax > 0 else 0
            bound = Fraction(P - 1, 2 ** 24) * mag + half_ulp
            assert abs(Fraction(float(xv[t, j])) - exact) <= bound, (t, j)


def test_negative_zero_partials_keep_their_sign():
    # every partial -0: -0 + -0 = -0, so x = -0 (a sum started from +0 would give +0).  With
    # n = 1 (alpha = 0) and h < 0, a = bf16(0 * h) = -0 and b = bf16(x_hat / 1) = -0, so h' = -0.
    P, T = 4, 2
    c = case(T=T, P=P, seed=9)
    parts = np.full((P, T, H), 0x8000, np.uint16)
    h = oracle.bf16_rne(-np.abs(oracle.bf16_to_f32(c["h"])) - 1.0)
    h_out, _, _, x = oracle.allreduce_boundary(h, parts, c["w_post"], c["w_pre"], 1,
                                               return_x=True)
    assert np.all(x == 0x8000)
    w_neg = (oracle.bf16_to_f32(c["w_post"]) < 0)
    assert np.all(h_out[:, ~w_neg] == 0x8000)
