"""Comparison helpers shared by the tests (no method arithmetic)."""
from __future__ import annotations

import numpy as np


def bf16_ordered(u: np.ndarray) -> np.ndarray:
    """Map BF16 bit patterns to integers ordered like their values (+0 and -0 both map to 0)."""
    u = np.asarray(u, dtype=np.uint16).astype(np.int32)
    return np.where(u & 0x8000, -(u & 0x7FFF), u)


def bf16_isnan(u: np.ndarray) -> np.ndarray:
    u = np.asarray(u, dtype=np.uint16)
    return ((u & 0x7F80) == 0x7F80) & ((u & 0x007F) != 0)


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """|a - b| in BF16 units in the last place; NaN vs NaN is 0, NaN vs number is a huge value."""
    a = np.asarray(a, dtype=np.uint16)
    b = np.asarray(b, dtype=np.uint16)
    d = np.abs(bf16_ordered(a) - bf16_ordered(b)).astype(np.int64)
    na, nb = bf16_isnan(a), bf16_isnan(b)
    d = np.where(na & nb, 0, d)
    d = np.where(na ^ nb, 1 << 30, d)
    return d


def f32_to_bf16_nearest(x: np.ndarray) -> np.ndarray:
    """Library rounding (torch, RNE) of float64/float32 values to BF16 bit patterns, used as an
    independent reference in pins."""
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def assert_bf16_close(got: np.ndarray, want: np.ndarray, max_ulp: int = 1,
                      min_equal: float = 0.999, what: str = "") -> None:
    """The parity bar: every element within ``max_ulp`` BF16 ulps and at least ``min_equal``
    of the elements bit-identical (NaN matches NaN)."""
    got = np.asarray(got, dtype=np.uint16).ravel()
    want = np.asarray(want, dtype=np.uint16).ravel()
    assert got.shape == want.shape, (got.shape, want.shape)
    if got.size == 0:
        return
    d = bf16_ulp_diff(got, want)
    worst = int(d.max())
    frac = float(np.mean(d == 0))
    assert worst <= max_ulp, f"{what}: max ulp diff {worst} at {int(d.argmax())} (> {max_ulp})"
    assert frac >= min_equal, f"{what}: only {frac:.6f} bit-identical (< {min_equal})"
