"""Pins of the oracle's BF16 round-to-nearest-even (CPU only).

The pages fix BF16 as the rounding type of the residual operands and the kernel outputs
("SGLang 支撑编程模型 Beam 生产部署", "三明治归一化与深度缩放残差"); the rounding rule is the
IEEE default, round to nearest with ties to even.  Pinned three ways: a hand-derived bit-pattern
table, the round trip of all 65,536 BF16 patterns, and agreement with torch's own FP32 -> BF16
conversion (a library RNE) on random FP32 bit patterns of every exponent.
"""
import os

import numpy as np
import torch

import oracle
from tests._util import bf16_isnan

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "bf16_rne_cases.txt")


def _cases():
    for line in open(GOLDEN, encoding="utf-8"):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        f_hex, want, *_ = line.split()
        yield int(f_hex, 16), want


def test_golden_bit_patterns():
    rows = list(_cases())
    assert len(rows) >= 20
    f = np.array([r[0] for r in rows], dtype=np.uint32).view(np.float32)
    got = oracle.bf16_rne(f)
    for (fbits, want), g in zip(rows, got):
        if want == "nan":
            assert bf16_isnan(np.uint16(g)), f"{fbits:08x} -> {int(g):04x}, want NaN"
        else:
            assert int(g) == int(want, 16), f"{fbits:08x} -> {int(g):04x}, want {want}"


def test_scalar_and_array_paths_agree():
    lib = oracle.lib()
    for fbits, _ in _cases():
        f = np.array([fbits], dtype=np.uint32).view(np.float32)
        assert lib.orc_bf16_rne(float(f[0])) == int(oracle.bf16_rne(f)[0]) or np.isnan(f[0])


def test_all_bf16_patterns_round_trip():
    b = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    f = oracle.bf16_to_f32(b)
    back = oracle.bf16_rne(f)
    nan = bf16_isnan(b)
    assert np.array_equal(back[~nan], b[~nan])
    assert bf16_isnan(back[nan]).all()


def test_matches_library_rne_on_random_fp32():
    g = np.random.Generator(np.random.PCG64(1234))
    bits = g.integers(0, 1 << 32, size=1 << 21, dtype=np.uint64).astype(np.uint32)
    # make ties and near-ties common: clear or set the low bits on a quarter each
    bits[: bits.size // 4] = (bits[: bits.size // 4] & 0xFFFF0000) | 0x8000
    bits[bits.size // 4: bits.size // 2] &= 0xFFFF8001
    f = bits.view(np.float32)
    got = oracle.bf16_rne(f)
    want = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(f)
    assert np.array_equal(got[~nan], want[~nan])
    assert bf16_isnan(got[nan]).all()
