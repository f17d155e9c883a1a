"""Helpers for the GPU parity tests: device placement, guard bands, launch-shape row counts."""
from __future__ import annotations

import numpy as np
import torch

import beam_inputs as bi
import residual_stream_norm_gb300 as rsn

CANARY = -12345.0  # exactly representable in BF16


def lib():
    rsn.build()
    return rsn.lib()


def dev(t: torch.Tensor) -> torch.Tensor:
    return t.to("cuda").contiguous()


class Guarded:
    """A device buffer with guard bands on both sides, filled with a canary; ``view`` is the
    usable region.  ``check()`` asserts the guards are untouched."""

    def __init__(self, shape, dtype=torch.bfloat16, guard=4096, fill=None):
        n = int(np.prod(shape))
        self.guard = guard
        self.buf = torch.full((n + 2 * guard,), CANARY, dtype=dtype, device="cuda")
        self.view = self.buf[guard: guard + n].view(*shape)
        if fill is not None:
            self.view.copy_(fill)

    def check(self):
        g = self.guard
        lo, hi = self.buf[:g], self.buf[-g:]
        assert bool((lo == CANARY).all()) and bool((hi == CANARY).all()), "guard band overwritten"


def persistent_T() -> int:
    """A row count just above the switch to the persistent kernels (4 rows per SM)."""
    return 4 * torch.cuda.get_device_properties(0).multi_processor_count + 5


def u16(t):
    return bi.u16(t)
