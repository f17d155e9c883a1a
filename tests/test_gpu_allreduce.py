"""GPU parity of beam_allreduce_boundary_fwd against the CPU oracle (needs a GB300).

The tensor-parallel all-reduce of the sublayer output fused ahead of the boundary chain ("Serving
Reflection Beam auf vLLM ab Tag 0", "Agentengetriebene Optimierung", change 3; "SGLang 支撑编程模型
Beam 生产部署", kernel-fusion paragraph).  The P partials sit in this GPU's memory.  Bar: every BF16
output within 1 ulp of the oracle and at least 99.9 % bit-identical; the FP32 per-token scales
within 2e-6 relative.
"""
import numpy as np
import pytest
import torch

import beam_inputs as bi
import oracle
import residual_stream_norm_gb300 as rsn
from tests._gpu import Guarded, dev, lib, persistent_T, u16
from tests._util import assert_bf16_close

pytestmark = pytest.mark.gpu

RSTD_RTOL = 2e-6


def run_gpu(c, parts=None, n=None):
    h = dev(c["h"])
    T, H = h.shape
    parts = dev(c["parts"]) if parts is None else parts
    h_out = torch.empty_like(h)
    y = torch.empty_like(h)
    rstd = torch.empty((T, 2), dtype=torch.float32, device="cuda")
    rsn.beam_allreduce_boundary_fwd(h_out, y, h, parts, dev(c["w_post"]), dev(c["w_pre"]),
                                    n or c["n"], bi.EPS, rstd)
    torch.cuda.synchronize()
    return u16(h_out), u16(y), rstd.cpu().numpy()


def oracle_run(c, n=None, threads=16):
    """The oracle over token slices on the host cores (rows are independent)."""
    h, p = u16(c["h"]), u16(c["parts"])
    wpo, wpr = u16(c["w_post"]), u16(c["w_pre"])
    T = h.shape[0]
    out = oracle.run_token_parallel(
        lambda lo, hi: oracle.allreduce_boundary(h[lo:hi], np.ascontiguousarray(p[:, lo:hi]),
                                                 wpo, wpr, n or c["n"]), T, threads)
    return tuple(np.concatenate([o[i] for o in out]) for i in range(3))


def check(got, want, what):
    assert_bf16_close(got[0], want[0], what=f"{what} h'")
    assert_bf16_close(got[1], want[1], what=f"{what} y")
    np.testing.assert_allclose(got[2], want[2], rtol=RSTD_RTOL, err_msg=f"{what} rstd")


def test_decode_tp8_boundaries():
    # batch-1 and T = 128 decode, TP8: the one-CTA-per-row kernel
    lib()
    for T, n in ((1, 1), (1, 57), (128, 104)):
        c = bi.allreduce_case(T=T, P=8, n=n, seed=T + n)
        check(run_gpu(c), oracle_run(c), f"T={T} n={n}")


@pytest.mark.parametrize("T,H,P", [
    (1, 8, 1), (3, 16, 2), (5, 5120, 3), (7, 5128, 8), (4, 16384, 8), (9, 5120, 16),
    (300, 5120, 8), (301, 4104, 5),
    # the persistent TMA ring (>= 4 rows per SM, at most 8 partials), ragged rows and the
    # per-row kernel for more than 8 partials or rows wider than 8 chunks
    (700, 5120, 8), (613, 5128, 1), (650, 1032, 3), (999, 6144, 7), (640, 4096, 2),
    (620, 16384, 8), (610, 5120, 16), (1500, 8, 8),
])
def test_shapes(T, H, P):
    c = bi.allreduce_case(T=T, H=H, P=P, n=(T * 7 + P) % 104 + 1, seed=T + H + P)
    check(run_gpu(c), oracle_run(c), f"T={T} H={H} P={P}")


def test_single_partial_equals_plain_boundary():
    # P = 1 is the plain boundary on that partial: bit-identical outputs
    for T in (5, 700):
        c = bi.allreduce_case(T=T, P=1, n=9, seed=T)
        got = run_gpu(c)
        h, x = dev(c["h"]), dev(c["parts"][0])
        h_out, y = torch.empty_like(h), torch.empty_like(h)
        rstd = torch.empty((T, 2), dtype=torch.float32, device="cuda")
        rsn.beam_boundary_fwd(h_out, y, h, x, dev(c["w_post"]), dev(c["w_pre"]), 9, bi.EPS, rstd)
        torch.cuda.synchronize()
        assert np.array_equal(got[0], u16(h_out)) and np.array_equal(got[1], u16(y))
        assert np.array_equal(got[2].view(np.uint32), rstd.cpu().numpy().view(np.uint32))


def test_rank_order_case_on_the_gpu():
    # partials (1, 2^-8, 2^-24, 2^-24) sum to the BF16 tie 1 + 2^-8 in rank order (rounds to 1)
    # and to 1 + 2^-8 + 2^-23 in reverse order (rounds up): the kernel must add in rank order
    T, H = 700, 5120
    vals = [1.0, 2.0 ** -8, 2.0 ** -24, 2.0 ** -24]
    for order in (vals, vals[::-1]):
        c = bi.allreduce_case(T=T, H=H, P=4, n=1, seed=3)
        c["parts"] = torch.stack([torch.full((T, H), v, dtype=torch.bfloat16) for v in order])
        check(run_gpu(c), oracle_run(c), f"order {order[0]}")


def test_repeated_buffer_and_y_aliasing_a_partial():
    # the same partial passed twice, and y written over rank 0's partial
    c = bi.allreduce_case(T=650, P=4, n=11, seed=5)
    parts = [dev(c["parts"][0]), dev(c["parts"][1]), dev(c["parts"][1]), dev(c["parts"][3])]
    want_c = dict(c, parts=torch.stack([c["parts"][0], c["parts"][1], c["parts"][1],
                                        c["parts"][3]]))
    want = oracle_run(want_c)
    h = dev(c["h"])
    rsn.beam_allreduce_boundary_fwd(h, parts[0], h, parts, dev(c["w_post"]), dev(c["w_pre"]), 11)
    torch.cuda.synchronize()
    assert_bf16_close(u16(h), want[0], what="in-place h'")
    assert_bf16_close(u16(parts[0]), want[1], what="y over rank 0's partial")


@pytest.mark.parametrize("which", ["rows", "persistent"])
def test_in_place_residual_with_guard_bands(which):
    # h' over h, with guard bands; "persistent" takes T = 4 SMs + 5 rows, just enough for the
    # persistent TMA ring
    T = 21 if which == "rows" else persistent_T()
    c = bi.allreduce_case(T=T, P=8, n=6, seed=T)
    H = c["h"].shape[1]
    want = oracle_run(c)
    h = Guarded((T, H), fill=dev(c["h"]))
    y = Guarded((T, H))
    rs = Guarded((T, 2), dtype=torch.float32)
    rsn.beam_allreduce_boundary_fwd(h.view, y.view, h.view, dev(c["parts"]), dev(c["w_post"]),
                                    dev(c["w_pre"]), 6, bi.EPS, rs.view)
    torch.cuda.synchronize()
    for g in (h, y, rs):
        g.check()
    check((u16(h.view), u16(y.view), rs.view.cpu().numpy()), want, f"in place T={T}")


def test_prefill_16384_tp8_every_row():
    # 8 x 2048 prefill, TP8, at the launch configuration the benchmark times: all rows compared
    c = bi.allreduce_case(T=16384, P=8, n=30, seed=16384)
    check(run_gpu(c), oracle_run(c), "prefill TP8")
    assert rsn.beam_device_faults() == 0


def test_zero_tokens():
    h = torch.empty((0, 5120), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(5120, dtype=torch.bfloat16, device="cuda")
    rsn.beam_allreduce_boundary_fwd(h, h, h, [h, h], w, w, 3)
    torch.cuda.synchronize()


@pytest.mark.parametrize("which", ["rows", "persistent"])
def test_nonfinite_overflowing_and_zero_partials(which):
    # NaN in one rank, +inf and -inf in others (separately, and meeting in one element: NaN), the
    # largest finite BF16 in every rank (the FP32 sum overflows to inf), all-zero and all -0
    # rows; the rest random.  IEEE results, as the oracle's.
    T = 8 if which == "rows" else persistent_T()
    c = bi.allreduce_case(T=T, P=4, n=5, seed=21)
    p = u16(c["parts"]).copy()
    p[0, 0, 3] = 0x7FC0                    # NaN
    p[1, 1, 7] = 0x7F80                    # +inf
    p[2, 1, 9] = 0xFF80                    # -inf
    p[1, 2, 11], p[3, 2, 11] = 0x7F80, 0xFF80   # +inf + -inf
    p[:, 3, :] = 0x7F7F                    # 4 x the largest finite BF16: inf in FP32
    p[:, 4, :] = 0                         # a zero row: r = 1/sqrt(eps)
    p[:, 5, :] = 0x8000                    # -0 in every rank
    p[:2, 6, :] = 0x5F34                   # two ranks of 1.3e19: squares near the FP32 top
    p[2:, 6, :] = 0
    c["parts"] = bi.from_u16(p)
    check(run_gpu(c), oracle_run(c), f"non-finite partials ({which})")
