"""Pins of the oracle's KV-cache write (CPU only).

The Q/K norm + RoPE kernel also writes K and V into the KV cache ("Serving Reflection Beam auf
vLLM ab Tag 0", section "MoE und Residual-Stream", change 6); the serving command runs an FP8
cache.  The oracle's FP8 E4M3 encoder is pinned against hand-derived codes, the round trip of
every code, and torch's float8_e4m3fn conversion; the cache write against closed forms.
"""
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp8_e4m3_cases.txt")


def _cases():
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        v, code, *_ = line.split()
        yield float(v), int(code, 16)


def test_fp8_golden_codes():
    n = 0
    for v, code in _cases():
        assert oracle.fp8_e4m3_rne(v) == code, (v, hex(code))
        n += 1
    assert n >= 25


def test_fp8_every_code_round_trips():
    for c in range(256):
        v = oracle.fp8_e4m3_to_f32(c)
        if (c & 0x7f) == 0x7f:
            assert np.isnan(v)
            continue
        assert oracle.fp8_e4m3_rne(v) == c, hex(c)
    # values grow with the code over the positive finite codes
    vals = [oracle.fp8_e4m3_to_f32(c) for c in range(0x7f)]
    assert all(a < b for a, b in zip(vals, vals[1:]))
    assert vals[-1] == 448.0 and vals[1] == 2.0 ** -9


def test_fp8_matches_torch_conversion_in_range():
    # torch rounds to nearest even as well; it has no saturation (|x| >= 464 gives NaN), so the
    # comparison stays below that
    g = np.random.default_rng(3)
    x = np.concatenate([g.uniform(-463.9, 463.9, 4000), g.normal(0, 1, 4000),
                        g.normal(0, 0.01, 2000), np.ldexp(g.uniform(-1, 1, 2000), -8)])
    x = x.astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([oracle.fp8_e4m3_rne(float(v)) for v in x], dtype=np.uint8)
    assert np.array_equal(got, want)


def _rows(T, nk, D, seed):
    g = np.random.default_rng(seed)
    k = g.normal(0, 1, (T, nk, D)).astype(np.float32)
    v = g.normal(0, 1, (T, nk, D)).astype(np.float32)
    return oracle.bf16_rne(k).reshape(T, nk, D), oracle.bf16_rne(v).reshape(T, nk, D)


def test_kv_cache_write_bf16_places_rows_and_skips_invalid_slots():
    T, nk, D, S = 6, 3, 16, 10
    k, v = _rows(T, nk, D, 1)
    slots = np.array([7, -1, 2, 10, 0, 5], np.int64)   # -1: padding; 10: out of range
    canary = np.full((S, nk, D), 0xABCD, np.uint16)
    kc, vc = oracle.kv_cache_write(canary, canary, k, v, slots, cache_dtype=0)
    for t, s in enumerate(slots):
        if 0 <= s < S:
            assert np.array_equal(kc[s], k[t]) and np.array_equal(vc[s], v[t])
    untouched = [s for s in range(S) if s not in set(slots.tolist())]
    assert all((kc[s] == 0xABCD).all() and (vc[s] == 0xABCD).all() for s in untouched)


def test_kv_cache_write_fp8_scales_then_encodes():
    T, nk, D, S = 4, 2, 8, 4
    k, v = _rows(T, nk, D, 2)
    slots = np.array([3, 1, 0, 2], np.int64)
    z = np.zeros((S, nk, D), np.uint8)
    kc, vc = oracle.kv_cache_write(z, z, k, v, slots, cache_dtype=1, k_scale=2.0, v_scale=0.5)
    kf = (k.astype(np.uint32) << 16).view(np.float32)
    vf = (v.astype(np.uint32) << 16).view(np.float32)
    for t, s in enumerate(slots):
        # k / 2 and v / 0.5 are exact: power-of-two scales
        want_k = [oracle.fp8_e4m3_rne(x / 2.0) for x in kf[t].ravel()]
        want_v = [oracle.fp8_e4m3_rne(x * 2.0) for x in vf[t].ravel()]
        assert kc[s].ravel().tolist() == want_k and vc[s].ravel().tolist() == want_v
    # scale 1: the code of each BF16 value, which decodes to that value's FP8 rounding
    kc1, _ = oracle.kv_cache_write(z, z, k, v, slots, cache_dtype=1)
    dec = np.array([oracle.fp8_e4m3_to_f32(c) for c in kc1[3].ravel()], np.float32)
    assert np.all(np.abs(dec - kf[0].ravel()) <= np.maximum(np.abs(kf[0].ravel()) / 16, 2.0 ** -10))
