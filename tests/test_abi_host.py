"""Host-side tests of the C ABI (no GPU needed).

The library must load on a machine without a GPU, export every entry point the header declares,
and reject every invalid argument with the documented status before any CUDA call -- these
calls never launch, so they run here with fake (never dereferenced) device addresses.
"""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from tests._util import f32_to_bf16_nearest
import residual_stream_norm_gb300 as rsn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beam_boundary.h")

OK, INVALID, MISALIGNED, UNSUPPORTED = 0, -1, -2, -3
A = 0x10000      # a 16-byte aligned fake device address (never dereferenced)
B = 0x20000
U = 0x30008      # 8-byte aligned only


@pytest.fixture(scope="module")
def lib():
    rsn.build()
    return rsn.lib()


def declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    return re.findall(r"BEAM_API\s+[\w\s\*]*?\b(beam_\w+)\s*\(", text)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) == 19, names
    raw = ctypes.CDLL(rsn.LIB_PATH)
    for nm in names:
        assert hasattr(raw, nm), f"{nm} declared in the header but not exported"


def test_version_and_status_strings(lib):
    assert rsn.beam_abi_version() == 2
    assert rsn.beam_status_str(0) == "BEAM_OK"
    assert rsn.beam_status_str(-2) == "BEAM_ERR_MISALIGNED"
    assert rsn.beam_status_str(42) == "unknown"


def test_residual_scales_match_oracle(lib):
    for n in list(range(1, 4097)) + [10**5, 2**20, 2**31 - 1]:
        assert rsn.beam_residual_scales(n) == oracle.residual_scales(n), n
    with pytest.raises(rsn.BeamError):
        rsn.beam_residual_scales(0)


def boundary(lib, h_out=A, y_out=B, h_in=A, x_in=B, wpo=A, wpr=B, T=4, H=5120, n=5, eps=1e-6,
             rstd=None):
    return lib.beam_boundary_fwd(h_out, y_out, h_in, x_in, wpo, wpr, T, H, n, eps, rstd, None)


@pytest.mark.parametrize("kw,want", [
    (dict(T=-1), INVALID), (dict(n=0), INVALID), (dict(H=0), INVALID), (dict(H=12), INVALID),
    (dict(H=16392), INVALID), (dict(eps=-1.0), INVALID), (dict(eps=float("nan")), INVALID),
    (dict(eps=float("inf")), INVALID), (dict(h_out=None), INVALID), (dict(x_in=None), INVALID),
    (dict(wpr=None), INVALID), (dict(h_in=A + 8), MISALIGNED), (dict(y_out=B + 2), MISALIGNED),
    (dict(wpo=A + 4), MISALIGNED), (dict(rstd=U + 4), MISALIGNED),
    (dict(T=0, h_out=None, y_out=None, h_in=None, x_in=None, wpo=None, wpr=None), OK),
])
def test_boundary_argument_checks(lib, kw, want):
    assert boundary(lib, **kw) == want


def moe(lib, K=8, topk=A, scale=2.5, T=4, e=B, **kw):
    return lib.beam_moe_combine_boundary_fwd(A, B, A, e, topk, scale, A, B, T, 5120, K, 5, 1e-6,
                                             None, None)


@pytest.mark.parametrize("kw,want", [
    (dict(K=0), INVALID), (dict(K=17), INVALID), (dict(scale=float("inf")), INVALID),
    (dict(topk=None), INVALID), (dict(e=None), INVALID), (dict(topk=A + 2), MISALIGNED),
    (dict(e=B + 8), MISALIGNED), (dict(T=0), OK),
])
def test_moe_argument_checks(lib, kw, want):
    assert moe(lib, **kw) == want


def allreduce(lib, parts=(A, B, A, B), P=None, T=4, H=5120, n=5, h_out=A, y_out=B,
              rstd=None):
    arr = (ctypes.c_void_p * max(1, len(parts)))(*parts)
    return lib.beam_allreduce_boundary_fwd(h_out, y_out, A, arr, len(parts) if P is None else P,
                                           A, B, T, H, n, 1e-6, rstd, None)


@pytest.mark.parametrize("kw,want", [
    (dict(P=0), INVALID), (dict(P=17), INVALID), (dict(T=-1), INVALID), (dict(n=0), INVALID),
    (dict(H=12), INVALID), (dict(parts=(A, None, B)), INVALID), (dict(h_out=None), INVALID),
    (dict(parts=(A, B + 8)), MISALIGNED), (dict(y_out=B + 2), MISALIGNED),
    (dict(rstd=U + 4), MISALIGNED), (dict(T=0), OK),
    # 16 partials (the same buffer may repeat) pass the checks; with T = 0 nothing launches
    (dict(parts=(A,) * 16, T=0), OK),
])
def test_allreduce_argument_checks(lib, kw, want):
    assert allreduce(lib, **kw) == want


def test_persistent_timeout_selftest_argument_checks(lib):
    f = lib.beam_selftest_persistent_timeout
    assert f(2, A, B, None, A, B, 4, 5120, 10**6, None) == INVALID      # kind
    assert f(0, A, B, None, A, B, 0, 5120, 10**6, None) == INVALID      # T
    assert f(0, A, B, None, A, B, 4, 16384, 10**6, None) == INVALID     # H > 8192
    assert f(1, A, B, None, A, B, 4, 5120, 10, None) == INVALID         # limit
    assert f(0, None, B, None, A, B, 4, 5120, 10**6, None) == INVALID
    assert f(0, A + 8, B, None, A, B, 4, 5120, 10**6, None) == MISALIGNED
    assert f(0, A, B, U + 4, A, B, 4, 5120, 10**6, None) == MISALIGNED


def qk(lib, fn="rope", q=A, k=B, qs=48 * 128, ks=8 * 128, pos=U, T=4, nq=48, nk=8, D=128,
       eps=1e-6, extra=(10000.0,)):
    f = lib.beam_qk_norm_rope_fwd if fn == "rope" else lib.beam_qk_norm_ssmax_fwd
    return f(q, k, qs, ks, A, B, pos, T, nq, nk, D, eps, *extra, None)


@pytest.mark.parametrize("fn,extra", [("rope", (10000.0,)), ("ssmax", (2048.0, 0.1))])
@pytest.mark.parametrize("kw,want", [
    (dict(D=64), UNSUPPORTED), (dict(D=256), UNSUPPORTED), (dict(T=-3), INVALID),
    (dict(nq=0, nk=0), INVALID), (dict(nq=-1), INVALID), (dict(nq=1000, nk=100), INVALID),
    (dict(pos=None), INVALID), (dict(q=None), INVALID), (dict(qs=48 * 128 - 8), INVALID),
    (dict(q=A + 8), MISALIGNED), (dict(qs=48 * 128 + 4), MISALIGNED),
    (dict(ks=8 * 128 + 2), MISALIGNED), (dict(pos=U + 4), MISALIGNED),
    (dict(T=0, q=None, k=None, pos=None), OK), (dict(nq=0, q=None, T=0), OK),
])
def test_qk_argument_checks(lib, fn, extra, kw, want):
    assert qk(lib, fn=fn, extra=extra, **kw) == want


def test_qk_parameter_checks(lib):
    assert qk(lib, fn="rope", extra=(0.0,)) == INVALID
    assert qk(lib, fn="rope", extra=(float("nan"),)) == INVALID
    assert qk(lib, fn="ssmax", extra=(0.0, 0.1)) == INVALID
    assert qk(lib, fn="ssmax", extra=(2048.0, float("inf"))) == INVALID


def qkv(lib, fn="rope", v=A, vs=8 * 128, slots=U, kc=A, vc=B, ns=64, dt=0, ksc=1.0, vsc=1.0,
        T=4, nq=48, nk=8, D=128, extra=(10000.0,)):
    f = lib.beam_qk_norm_rope_kv_fwd if fn == "rope" else lib.beam_qk_norm_ssmax_kv_fwd
    return f(A, B, 48 * 128, 8 * 128, v, vs, A, B, U, slots, kc, vc, ns, dt, ksc, vsc, T, nq, nk,
             D, 1e-6, *extra, None)


@pytest.mark.parametrize("fn,extra", [("rope", (10000.0,)), ("ssmax", (2048.0, 0.1))])
@pytest.mark.parametrize("kw,want", [
    (dict(dt=2), UNSUPPORTED), (dict(dt=-1), UNSUPPORTED), (dict(ns=-1), INVALID),
    (dict(v=None), INVALID), (dict(slots=None), INVALID), (dict(kc=None), INVALID),
    (dict(vc=None), INVALID), (dict(vs=8 * 128 - 8), INVALID),
    (dict(dt=1, ksc=0.0), INVALID), (dict(dt=1, vsc=float("inf")), INVALID),
    (dict(dt=1, ksc=-2.0), INVALID), (dict(v=A + 8), MISALIGNED),
    (dict(vs=8 * 128 + 4), MISALIGNED), (dict(slots=U + 4), MISALIGNED),
    (dict(kc=A + 8), MISALIGNED), (dict(dt=1, vc=B + 4), MISALIGNED),
    (dict(T=0, v=None, slots=None, kc=None, vc=None), OK),
])
def test_qk_kv_argument_checks(lib, fn, extra, kw, want):
    assert qkv(lib, fn=fn, extra=extra, **kw) == want


def gate(lib, out=A, attn=A, g=B, bias=U, T=4, nh=48, D=128, sa=6144, sg=6144, so=6144):
    return lib.beam_attn_gate_fwd(out, attn, g, bias, T, nh, D, sa, sg, so, None)


@pytest.mark.parametrize("kw,want", [
    (dict(D=12), UNSUPPORTED), (dict(D=0), UNSUPPORTED), (dict(D=2048), UNSUPPORTED),
    (dict(nh=0), INVALID), (dict(T=-1), INVALID), (dict(bias=None), INVALID),
    (dict(sa=6136), INVALID), (dict(out=A + 8), MISALIGNED), (dict(bias=U + 2), MISALIGNED),
    (dict(sg=6148), MISALIGNED), (dict(T=0, out=None, attn=None, g=None, bias=None), OK),
])
def test_gate_argument_checks(lib, kw, want):
    assert gate(lib, **kw) == want


def test_rejected_calls_raise_in_the_binding(lib):
    with pytest.raises(rsn.BeamError) as e:
        rsn._call("beam_boundary_fwd", A, B, A, B, A, B, 4, 12, 5, 1e-6, None, None)
    assert e.value.status == INVALID


# ------------------------------------------------------------------------------------------
# the RoPE cos / sin routine (host build of the device code)
# ------------------------------------------------------------------------------------------

def _rounded(x32):
    x = x32.astype(np.float64)
    return np.cos(x).astype(np.float32), np.sin(x).astype(np.float32)


def _check_rounded(angles, what, tiny=2.0 ** -20):
    c, s = rsn.beam_rope_cos_sin(angles)
    wc, ws = _rounded(angles)
    for got, want in ((c, wc), (s, ws)):
        bad = got != want
        # a miss may only be a near tie of a tiny value (whose absolute error is ~2^-47)
        assert not np.any(bad & (np.abs(want) >= tiny)), (what, angles[bad][:5], got[bad][:5],
                                                          want[bad][:5])
        assert np.mean(bad) < 1e-6, (what, np.mean(bad))
        if np.any(bad):
            ulps = np.abs(got[bad].view(np.int32).astype(np.int64) -
                          want[bad].view(np.int32).astype(np.int64))
            assert ulps.max() <= 1


def test_rope_cos_sin_on_all_kernel_angles(lib):
    # every frequency of head_dim 128 at theta 1e4 and 5e5, positions sampled over [0, 2^20)
    # and near 2^24: angle = fp32(fp32(pos) * fp32(theta^(-2i/128)))
    for theta in (10000.0, 500000.0):
        inv = oracle.rope_inv_freq(theta, 128)
        pos = np.concatenate([np.arange(0, 1 << 20, 37), np.arange((1 << 24) - 4096, 1 << 24, 3)])
        ang = (pos.astype(np.float32)[:, None] * inv[None, :]).astype(np.float32).ravel()
        _check_rounded(ang, f"theta={theta}")


def test_rope_cos_sin_random_fp32(lib):
    g = np.random.Generator(np.random.PCG64(7))
    e = g.uniform(-30, 24, size=1 << 21)
    x = (np.sign(g.uniform(-1, 1, size=e.size)) * 2.0 ** e).astype(np.float32)
    x = x[np.abs(x) < 2 ** 24]
    _check_rounded(x, "random")
    # special values and neighbours of multiples of pi/2
    k = np.arange(-2000, 2000, dtype=np.float64)
    near = (k * np.pi / 2).astype(np.float32)
    near = np.concatenate([near, np.nextafter(near, np.float32(np.inf)),
                           np.nextafter(near, np.float32(-np.inf)),
                           np.array([0.0, -0.0, 1e-30, -1e-30, 0.5, 1.0], np.float32)])
    _check_rounded(near.astype(np.float32), "near k*pi/2")
    c, s = rsn.beam_rope_cos_sin(np.array([0.0, -0.0], np.float32))
    assert np.all(c == 1.0) and s[0] == 0.0 and np.signbit(s[1])


def test_rope_cos_sin_rejects_out_of_range(lib):
    with pytest.raises(rsn.BeamError):
        rsn.beam_rope_cos_sin(np.array([2.0 ** 24], np.float32))
    with pytest.raises(rsn.BeamError):
        rsn.beam_rope_cos_sin(np.array([np.nan], np.float32))


# ------------------------------------------------------------------------------------------
# the residual operand division (host build of the kernels' arithmetic)
# ------------------------------------------------------------------------------------------

def _bf16_values(finite_only=True):
    b = np.arange(1 << 16, dtype=np.uint32)
    x = (b << 16).view(np.float32)
    return x[np.isfinite(x)] if finite_only else x[~np.isnan(x)]


def _bf16_of_ieee_quotient(x, n):
    s = np.float32(np.sqrt(np.float64(n)))
    return f32_to_bf16_nearest(x / s)


def _bits(b):
    return (b.view(np.uint32) >> 16).astype(np.uint16)


def test_residual_operand_equals_bf16_of_ieee_division_exhaustively(lib):
    # every BF16 value x (subnormals, signed zeros and infinities included) and every residual
    # index n = 1..4096: the kernels' b must be bf16 of the IEEE (correctly rounded) FP32
    # quotient -- whichever of the product or the division the kernels' rule picks.
    x = _bf16_values(finite_only=False)
    for n in range(1, 4097):
        b = rsn.beam_residual_operand(x, n)
        want = _bf16_of_ieee_quotient(x, n)
        assert np.array_equal(_bits(b), want), n


def test_residual_operand_large_n_nan_and_non_bf16_inputs(lib):
    x = _bf16_values(finite_only=False)
    for n in (4097, 10**5, 10**6 + 3, 2**24, 2**31 - 1):
        b = rsn.beam_residual_operand(x, n)
        assert np.array_equal(_bits(b), _bf16_of_ieee_quotient(x, n)), n
    assert np.isnan(rsn.beam_residual_operand(np.array([np.nan], np.float32), 5)).all()
    with pytest.raises(rsn.BeamError):  # 1 + 2^-20 is not a BF16 value
        rsn.beam_residual_operand(np.array([1.0 + 2.0**-20], np.float32), 5)
    with pytest.raises(rsn.BeamError):
        rsn.beam_residual_operand(np.array([1.0], np.float32), 0)


# ------------------------------------------------------------------------------------------
# the kernels' rare exact path for sums of squares (host build of the same integer code)
# ------------------------------------------------------------------------------------------

def _as_bf16(x):
    """float32 values rounded to BF16 (nearest even), returned as float32."""
    bits = f32_to_bf16_nearest(np.asarray(x, dtype=np.float64)).astype(np.uint32) << 16
    return bits.view(np.float32)


def _check_exact_square_sum(v):
    v = np.asarray(v, dtype=np.float32)
    got = rsn.beam_exact_square_sum(v)
    with np.errstate(over="ignore", invalid="ignore"):
        want = oracle.exact_sum_f32(v * v)
    if np.isnan(want):
        assert np.isnan(got)
    else:
        assert np.float32(got).view(np.uint32) == np.float32(want).view(np.uint32), (got, want)


def test_exact_square_sum_matches_exact_rounding_on_beam_rows(lib):
    # rows like the boundary's inputs: N(0,1) * s_t, s_t ~ U(0.5, 4), some with x16 outliers
    g = np.random.default_rng(11)
    for k in range(400):
        n = int(g.choice([128, 5120, 16384]))
        v = g.standard_normal(n) * g.uniform(0.5, 4.0)
        if k % 7 == 0:
            v[g.integers(0, n, 4)] *= 16.0
        _check_exact_square_sum(_as_bf16(v))


def test_exact_square_sum_wide_ranges_tiny_and_huge(lib):
    g = np.random.default_rng(12)
    for k in range(200):
        n = int(g.integers(1, 600))
        e = g.integers(-70, 64, n) if k % 2 else g.integers(-20, 20, n)  # squares 2^-140 .. 2^128
        v = np.ldexp(g.uniform(1.0, 2.0, n), e) * g.choice([-1.0, 1.0], n)
        _check_exact_square_sum(_as_bf16(v))
    # subnormal squares and subnormal sums
    _check_exact_square_sum(_as_bf16(np.ldexp(np.ones(37), -70)))
    _check_exact_square_sum(_as_bf16(np.ldexp(g.uniform(1, 2, 300), -66)))
    # overflow of a square and of the sum
    _check_exact_square_sum(np.array([2.0 ** 64, 1.0], np.float32))
    _check_exact_square_sum(_as_bf16(np.full(5120, 2.0 ** 63)))
    # zeros, NaN, one element
    _check_exact_square_sum(np.zeros(17, np.float32))
    _check_exact_square_sum(np.array([1.0, np.nan, 2.0], np.float32))
    _check_exact_square_sum(np.array([-3.0], np.float32))
    assert rsn.beam_exact_square_sum(np.zeros(0, np.float32)) == 0.0


def test_exact_square_sum_rounds_ties_to_even_and_breaks_them_with_tiny_terms(lib):
    # 1 + 2^-24 is the midpoint between 1 and 1 + 2^-23: ties to even (1.0)
    assert rsn.beam_exact_square_sum(np.array([1.0, 2.0 ** -12], np.float32)) == 1.0
    # a term far below the accumulator's range still breaks the tie upwards (sticky)
    up = np.float32(1.0 + 2.0 ** -23)
    for tiny in (2.0 ** -30, 2.0 ** -50, 2.0 ** -70):
        v = np.array([1.0, 2.0 ** -12, tiny], np.float32)
        assert rsn.beam_exact_square_sum(v) == up, tiny
        _check_exact_square_sum(v)
    # 1 + 3 * 2^-24 is the midpoint above 1 + 2^-23 (odd): ties to even rounds up
    v = np.array([1.0, 2.0 ** -12, 2.0 ** -12, 2.0 ** -12], np.float32)
    _check_exact_square_sum(v)


def test_exact_square_sum_argument_checks(lib):
    with pytest.raises(rsn.BeamError):
        rsn.beam_exact_square_sum(np.zeros(16385, np.float32))


# ------------------------------------------------------------------------------------------
# the routing sigmoid (host build of the kernels' arithmetic) and the routing call's checks
# ------------------------------------------------------------------------------------------

def test_routing_sigmoid_equals_the_oracle_on_a_sweep(lib):
    # every 512th FP32 pattern over the range where the sigmoid is neither 0 nor 1 by overflow,
    # plus random and edge values: bit-identical to the oracle's long-double evaluation
    u = np.arange(0, 1 << 32, 512, dtype=np.uint64).astype(np.uint32)
    z = u.view(np.float32)
    z = z[np.isfinite(z) & (z > -89.5) & (z < 18.0)]
    edges = np.array([0.0, -0.0, 16.9, 17.0, 17.1, -88.72, -88.7228, -88.73, -89.0, -100.0,
                      100.0, 1e-30, -1e-30, np.inf, -np.inf], np.float32)
    g = np.random.default_rng(9)
    z = np.concatenate([z, edges, g.normal(0, 3, 200000).astype(np.float32)])
    got = rsn.beam_routing_sigmoid(z)
    want = oracle.sigmoid_array(z)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert np.isnan(rsn.beam_routing_sigmoid(np.array([np.nan], np.float32))).all()


def route(lib, ids=A, w=B, logits=A + 4096, bias=B + 4096, T=4, E=256, G=8, TG=4, K=8):
    return lib.beam_grouped_topk_fwd(ids, w, logits, bias, T, E, G, TG, K, None)


@pytest.mark.parametrize("kw,want", [
    (dict(E=128), UNSUPPORTED), (dict(G=4), UNSUPPORTED), (dict(TG=3), UNSUPPORTED),
    (dict(K=6), UNSUPPORTED), (dict(T=-1), INVALID), (dict(ids=None), INVALID),
    (dict(w=None), INVALID), (dict(logits=None), INVALID), (dict(bias=None), INVALID),
    (dict(logits=A + 8), MISALIGNED), (dict(bias=B + 8), MISALIGNED),
    (dict(ids=A + 2), MISALIGNED),
    (dict(T=0, ids=None, w=None, logits=None, bias=None), OK),
])
def test_routing_argument_checks(lib, kw, want):
    assert route(lib, **kw) == want


def test_selftest_copy_timeout_limit_checks(lib):
    assert lib.beam_selftest_copy_timeout(10, None) == INVALID
    assert lib.beam_selftest_copy_timeout(3_000_000_000, None) == INVALID
