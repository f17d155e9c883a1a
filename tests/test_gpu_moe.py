"""GPU parity of beam_moe_combine_boundary_fwd against the CPU oracle (needs a GB300).

Top-K expert combine with FP32 renormalised weights times 2.5, fused ahead of the boundary chain
("Serving Reflection Beam auf vLLM ab Tag 0": "MoE und Residual-Stream", bullet "MoE im
DeepSeek-V3-Stil"; "Agentengetriebene Optimierung", change 3).
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


def run_gpu(h, e, w, w_post, w_pre, n, scale=bi.ROUTED_SCALING, eps=bi.EPS):
    T, K, H = e.shape
    h_out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(h_out)
    rstd = torch.empty((T, 2), dtype=torch.float32, device="cuda")
    rsn.beam_moe_combine_boundary_fwd(h_out, y, dev(h), dev(e), dev(w), dev(w_post), dev(w_pre),
                                      n, eps, scale, rstd)
    torch.cuda.synchronize()
    return u16(h_out), u16(y), rstd.cpu().numpy()


def oracle_run(c, n=None, scale=bi.ROUTED_SCALING):
    return oracle.moe_combine_boundary(u16(c["h"]), u16(c["e"]), c["topk_w"].numpy(),
                                       u16(c["w_post"]), u16(c["w_pre"]), n or c["n"],
                                       routed_scaling=scale)


def check(got, want, what):
    assert_bf16_close(got[0], want[0], what=f"{what} h'")
    assert_bf16_close(got[1], want[1], what=f"{what} y")
    np.testing.assert_allclose(got[2], want[2], rtol=2e-6, err_msg=f"{what} rstd")


def test_decode_moe_boundaries_layers_3_to_51():
    # T = 128 decode, top-8 of [128, 8, 5120]; one launch per MoE layer 3..51 with its own
    # residual index n = 2*layer + 2 and its own norm weights.
    lib()
    base = bi.moe_case(T=128, seed=0)
    e, w, h = dev(base["e"]), dev(base["topk_w"]), dev(base["h"])
    g = bi.rng(99)
    for layer in range(3, 52):
        n = 2 * layer + 2
        wpo, wpr = bi.norm_weight(g, bi.HIDDEN), bi.norm_weight(g, bi.HIDDEN)
        h_out = torch.empty_like(h)
        y = torch.empty_like(h)
        rsn.beam_moe_combine_boundary_fwd(h_out, y, h, e, w, dev(wpo), dev(wpr), n)
        torch.cuda.synchronize()
        want = oracle.moe_combine_boundary(u16(base["h"]), u16(base["e"]),
                                           base["topk_w"].numpy(), u16(wpo), u16(wpr), n)
        assert_bf16_close(u16(h_out), want[0], what=f"layer {layer} h'")
        assert_bf16_close(u16(y), want[1], what=f"layer {layer} y")


@pytest.mark.parametrize("T,H,K", [(1, 8, 1), (3, 16, 3), (5, 5120, 16), (2, 5128, 8),
                                   (310, 5120, 8), (4, 16384, 8), (300, 16384, 2),
                                   # persistent TMA ring (>= 4 rows per SM), and shapes whose
                                   # stages do not fit shared memory (per-row fallback)
                                   (700, 5120, 8), (650, 5128, 1), (620, 16384, 2),
                                   (610, 5120, 16), (900, 16384, 8), (1500, 8, 8),
                                   # the 3-stage ring with fewer slots and other row widths
                                   (700, 1032, 3), (640, 4096, 8), (999, 6144, 7)])
def test_shapes(T, H, K):
    c = bi.moe_case(T=T, H=H, K=K, seed=T * 7 + K)
    check(run_gpu(c["h"], c["e"], c["topk_w"], c["w_post"], c["w_pre"], c["n"]), oracle_run(c),
          f"T={T} H={H} K={K}")


def test_scale_and_weight_variants():
    c = bi.moe_case(T=16, seed=5)
    for scale in (1.0, 2.5, -0.75):
        check(run_gpu(c["h"], c["e"], c["topk_w"], c["w_post"], c["w_pre"], 9, scale=scale),
              oracle_run(c, n=9, scale=scale), f"scale={scale}")
    w = torch.zeros_like(c["topk_w"])
    w[:, 3] = 1.0  # one-hot
    c1 = dict(c, topk_w=w)
    check(run_gpu(c["h"], c["e"], w, c["w_post"], c["w_pre"], 9), oracle_run(c1, n=9), "one-hot")


def test_prefill_16384_every_row():
    # 8 x 2048 prefill MoE variant, full size: e [16384, 8, 5120] (1.34 GB); the oracle recomputes
    # every row (token slices on the host cores).
    c = bi.moe_case(T=16384, seed=1)
    T = 16384
    h = dev(c["h"])
    e, w = dev(c["e"]), dev(c["topk_w"])
    h_out = torch.empty_like(h)
    y = torch.empty_like(h)
    rstd = torch.empty((T, 2), dtype=torch.float32, device="cuda")
    rsn.beam_moe_combine_boundary_fwd(h_out, y, h, e, w, dev(c["w_post"]), dev(c["w_pre"]),
                                      c["n"], bi.EPS, bi.ROUTED_SCALING, rstd)
    torch.cuda.synchronize()
    hu, eu, wn = u16(c["h"]), u16(c["e"]), c["topk_w"].numpy()
    wpo, wpr = u16(c["w_post"]), u16(c["w_pre"])
    parts = oracle.run_token_parallel(
        lambda lo, hi: oracle.moe_combine_boundary(hu[lo:hi], eu[lo:hi], wn[lo:hi], wpo, wpr,
                                                   c["n"]), T, 16)
    want = tuple(np.concatenate([p[i] for p in parts]) for i in range(3))
    check((u16(h_out), u16(y), rstd.cpu().numpy()), want, "prefill MoE")


@pytest.mark.parametrize("which", ["rows", "persistent"])
def test_in_place_residual_and_guards(which):
    # h' over h with guard bands; "persistent" takes T = 4 SMs + 5 rows, just enough for the TMA
    # ring, whose producer copies later rows while the consumers write earlier ones back
    T = 21 if which == "rows" else persistent_T()
    c = bi.moe_case(T=T, seed=6)
    _, K, H = c["e"].shape
    want = oracle_run(c)
    h = Guarded((T, H), fill=dev(c["h"]))
    y = Guarded((T, H))
    rsn.beam_moe_combine_boundary_fwd(h.view, y.view, h.view, dev(c["e"]), dev(c["topk_w"]),
                                      dev(c["w_post"]), dev(c["w_pre"]), c["n"])
    torch.cuda.synchronize()
    h.check()
    y.check()
    assert_bf16_close(u16(h.view), want[0], what=f"in-place h' ({which})")
    assert_bf16_close(u16(y.view), want[1], what=f"y ({which})")


def test_zero_tokens():
    e = torch.empty((0, 8, 5120), dtype=torch.bfloat16, device="cuda")
    h = torch.empty((0, 5120), dtype=torch.bfloat16, device="cuda")
    w = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    wn = torch.ones(5120, dtype=torch.bfloat16, device="cuda")
    rsn.beam_moe_combine_boundary_fwd(h, h, h, e, w, wn, wn, 8)
    torch.cuda.synchronize()
