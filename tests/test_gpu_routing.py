"""GPU parity of the grouped top-k routing against the CPU oracle (needs a GB300).

Beam routes its 256 experts like DeepSeek-V3 ("Serving Reflection Beam auf vLLM ab Tag 0",
section "MoE und Residual-Stream", bullets "MoE im DeepSeek-V3-Stil", "FP32-Router"; "SGLang 支撑
编程模型 Beam 生产部署", "稠密层与分组 MoE 路由").  Every sigmoid is the correctly rounded FP32
value on both sides, so expert ids and weights are compared bit for bit.
"""
import numpy as np
import pytest
import torch

import beam_inputs as bi
import oracle
import residual_stream_norm_gb300 as rsn
from tests._gpu import dev, lib, u16
from tests._util import assert_bf16_close

pytestmark = pytest.mark.gpu


def run(logits, bias):
    T = logits.shape[0]
    ids = torch.full((T, 8), -7, dtype=torch.int32, device="cuda")
    w = torch.full((T, 8), -1.0, dtype=torch.float32, device="cuda")
    rsn.beam_grouped_topk_fwd(ids, w, dev(logits), dev(bias))
    torch.cuda.synchronize()
    return ids.cpu().numpy(), w.cpu().numpy()


def check(logits, bias, what):
    gi, gw = run(logits, bias)
    oi, ow = oracle.grouped_topk(logits.numpy(), bias.numpy())
    bad = np.nonzero((gi != oi).any(1))[0][:8]
    assert np.array_equal(gi, oi), f"{what}: ids differ at tokens {bad}"
    assert np.array_equal(gw.view(np.uint32), ow.view(np.uint32)), f"{what}: weights differ"


@pytest.mark.parametrize("T", [1, 128, 2048, 16384])
def test_routing_configs(T):
    lib()
    c = bi.routing_case(T=T, seed=T)
    check(c["logits"], c["bias"], f"T={T}")


@pytest.mark.parametrize("std", [0.05, 4.0, 30.0])
def test_routing_logit_scales(std):
    # near-equal scores (small spread: many near ties) and saturated sigmoids (large spread:
    # many scores exactly 0 or 1, ties broken by index)
    c = bi.routing_case(T=700, seed=11, logit_std=std)
    check(c["logits"], c["bias"], f"std={std}")


def test_routing_ties_nan_and_infinities():
    T = 64
    g = np.random.default_rng(4)
    z = np.zeros((T, 256), np.float32)
    z[1] = 3.0                                      # all equal: groups 0..3, experts 0..7
    z[2, ::7] = np.nan                              # NaN ranks last
    z[3, :] = np.inf                                # every score exactly 1
    z[4, :] = -np.inf                               # every score exactly 0: weights 0/0 = NaN
    z[5, :128] = 50.0                               # saturated half
    z[6, g.integers(0, 256, 40)] = np.nan
    z[7:] = g.normal(0, 2, (T - 7, 256)).astype(np.float32)
    b = np.zeros(256, np.float32)
    b[200:] = 0.25
    gi, gw = run(torch.from_numpy(z), torch.from_numpy(b))
    oi, ow = oracle.grouped_topk(z, b)
    assert np.array_equal(gi, oi)
    both_nan = np.isnan(gw) & np.isnan(ow)
    assert np.array_equal(np.where(both_nan, 0, gw).view(np.uint32),
                          np.where(both_nan, 0, ow).view(np.uint32))


def test_routing_feeds_the_moe_combine():
    # the routing weights drive the combine boundary: GPU routing -> GPU combine equals oracle
    # routing -> oracle combine
    T = 96
    c = bi.routing_case(T=T, seed=21)
    m = bi.moe_case(T=T, seed=22)
    gi, gw = run(c["logits"], c["bias"])
    h_out = torch.empty_like(dev(m["h"]))
    y = torch.empty_like(h_out)
    rsn.beam_moe_combine_boundary_fwd(h_out, y, dev(m["h"]), dev(m["e"]),
                                      torch.from_numpy(gw).cuda(), dev(m["w_post"]),
                                      dev(m["w_pre"]), m["n"], bi.EPS, bi.ROUTED_SCALING)
    torch.cuda.synchronize()
    oi, ow = oracle.grouped_topk(c["logits"].numpy(), c["bias"].numpy())
    wh, wy, _ = oracle.moe_combine_boundary(u16(m["h"]), u16(m["e"]), ow, u16(m["w_post"]),
                                            u16(m["w_pre"]), m["n"], bi.EPS, bi.ROUTED_SCALING)
    assert np.array_equal(gi, oi)
    assert_bf16_close(u16(h_out), wh, what="routed combine h'")
    assert_bf16_close(u16(y), wy, what="routed combine y")


def test_routing_zero_tokens():
    ids = torch.empty((0, 8), dtype=torch.int32, device="cuda")
    w = torch.empty((0, 8), dtype=torch.float32, device="cuda")
    rsn.beam_grouped_topk_fwd(ids, w, torch.empty((0, 256), device="cuda"),
                              torch.zeros(256, device="cuda"))
    torch.cuda.synchronize()
