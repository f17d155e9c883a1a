"""GPU parity of the Q/K kernels fused with the KV-cache write (needs a GB300).

"Serving Reflection Beam auf vLLM ab Tag 0", section "MoE und Residual-Stream", change 6: the
Q/K-norm and RoPE kernel also writes K and V into the KV cache; the serving command runs an FP8
cache.  The oracle is the unfused pipeline: the Q/K norm (+ RoPE or SSMax), then the cache
write of the stored K' and of V (oracle.kv_cache_write).
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
D = bi.HEAD_DIM
GUARD = 4096


class GuardedCache:
    """A cache [num_slots, nk, 128] in the middle of a buffer filled with a canary byte pattern;
    check() asserts that the guard bands are untouched."""

    def __init__(self, num_slots, nk, fp8):
        self.fp8 = fp8
        esz = 1 if fp8 else 2
        n = num_slots * nk * D * esz
        self.buf = torch.full((n + 2 * GUARD,), 0xA5, dtype=torch.uint8, device="cuda")
        body = self.buf[GUARD: GUARD + n]
        self.view = body.view(num_slots, nk, D) if fp8 else \
            body.view(torch.bfloat16).view(num_slots, nk, D)

    def host(self):
        t = self.view.cpu()
        return t.numpy() if self.fp8 else t.view(torch.int16).numpy().view(np.uint16)

    def check(self):
        assert bool((self.buf[:GUARD] == 0xA5).all()) and bool((self.buf[-GUARD:] == 0xA5).all())


def run(kind, c, kv, fp8, k_scale=1.0, v_scale=1.0, q=None, k=None, v=None):
    nk = c["k"].shape[1]
    kc = GuardedCache(kv["num_slots"], nk, fp8)
    vc = GuardedCache(kv["num_slots"], nk, fp8)
    init_k, init_v = kc.host(), vc.host()
    q = dev(c["q"]) if q is None else q
    k = dev(c["k"]) if k is None else k
    v = dev(kv["v"]) if v is None else v
    fn = rsn.beam_qk_norm_rope_kv_fwd if kind == "rope" else rsn.beam_qk_norm_ssmax_kv_fwd
    fn(q, k, v, dev(c["wq"]), dev(c["wk"]), dev(c["pos"]), dev(kv["slot_mapping"]), kc.view,
       vc.view, cache_dtype=rsn.CACHE_FP8_E4M3 if fp8 else rsn.CACHE_BF16, k_scale=k_scale,
       v_scale=v_scale)
    torch.cuda.synchronize()
    kc.check()
    vc.check()
    return q, k, kc.host(), vc.host(), init_k, init_v


def oracle_all(kind, c, kv, fp8, init_k, init_v, k_scale=1.0, v_scale=1.0):
    fo = oracle.qk_norm_rope if kind == "rope" else oracle.qk_norm_ssmax
    wq, wk = fo(u16(c["q"]), u16(c["k"]), u16(c["wq"]), u16(c["wk"]), c["pos"].numpy())
    kc, vc = oracle.kv_cache_write(init_k, init_v, wk, u16(kv["v"]), kv["slot_mapping"].numpy(),
                                   cache_dtype=1 if fp8 else 0, k_scale=k_scale, v_scale=v_scale)
    return wq, wk, kc, vc


def check_caches(kind, c, kv, fp8, got, k_scale=1.0, v_scale=1.0, what=""):
    q, k, gkc, gvc, init_k, init_v = got
    wq, wk, okc, ovc = oracle_all(kind, c, kv, fp8, init_k, init_v, k_scale, v_scale)
    assert_bf16_close(u16(q), wq, what=f"{what} q")
    assert_bf16_close(u16(k), wk, what=f"{what} k")
    # V is copied (or encoded) as it is: bit-exact against the oracle everywhere, untouched
    # slots included
    assert np.array_equal(gvc, ovc), f"{what} v cache"
    # the K cache holds the stored K': bit-exact against the cache write of the GPU's own K'
    # (K' itself is within the parity bar of the oracle's, checked above)
    mk, _ = oracle.kv_cache_write(init_k, init_v, u16(k), u16(kv["v"]),
                                  kv["slot_mapping"].numpy(), cache_dtype=1 if fp8 else 0,
                                  k_scale=k_scale, v_scale=v_scale)
    assert np.array_equal(gkc, mk), f"{what} k cache"
    if kind == "rope":  # RoPE outputs are bit-identical to the oracle's, so is the cache
        assert np.array_equal(gkc, okc), f"{what} k cache vs oracle"


@pytest.mark.parametrize("kind", ["rope", "ssmax"])
@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("T,mode", [(128, "uniform"), (2048, "contiguous"), (1999, "uniform"),
                                    (4901, "uniform")])
def test_qk_kv_configs(kind, fp8, T, mode):
    lib()
    c = bi.attn_qk_case(T=T, seed=T + 1, pos_mode=mode)
    kv = bi.kv_cache_case(T=T, seed=T + 2)
    check_caches(kind, c, kv, fp8, run(kind, c, kv, fp8), what=f"{kind} fp8={fp8} T={T}")


@pytest.mark.parametrize("kind", ["rope", "ssmax"])
@pytest.mark.parametrize("k_scale,v_scale", [(0.5, 4.0), (3.0, 0.3)])
@pytest.mark.parametrize("T", [64, 1001, 4901])
def test_fp8_scales_power_of_two_and_general(kind, k_scale, v_scale, T):
    # T = 1001: the staged kernel, with a ragged last tile
    c = bi.attn_qk_case(T=T, seed=5)
    kv = bi.kv_cache_case(T=T, seed=6)
    got = run(kind, c, kv, True, k_scale, v_scale)
    check_caches(kind, c, kv, True, got, k_scale, v_scale,
                 what=f"scales {k_scale},{v_scale} T={T}")


@pytest.mark.parametrize("T", [9, 1001, 4901])
@pytest.mark.parametrize("nq,nk", [(1, 1), (3, 2), (64, 8), (0, 3), (5, 0)])
def test_head_counts_with_cache(nq, nk, T):
    c = bi.attn_qk_case(T=T, n_q=nq, n_kv=nk, seed=nq * 7 + nk)
    kv = bi.kv_cache_case(T=T, n_kv=nk, seed=3, pad_frac=0.2, oob_frac=0.1)
    q = dev(c["q"]) if nq else torch.empty((T, 0, D), dtype=torch.bfloat16, device="cuda")
    k = dev(c["k"]) if nk else torch.empty((T, 0, D), dtype=torch.bfloat16, device="cuda")
    v = dev(kv["v"]) if nk else torch.empty((T, 0, D), dtype=torch.bfloat16, device="cuda")
    for fp8 in (False, True):
        got = run("rope", c, kv, fp8, q=q.clone(), k=k.clone(), v=v)
        check_caches("rope", c, kv, fp8, got, what=f"{nq}/{nk} fp8={fp8}")


@pytest.mark.parametrize("T", [33, 1001, 4901])
def test_views_into_packed_qkv_projection(T):
    # Q, K and V as row-strided views of one packed [T, (48 + 8 + 8) * 128] projection output
    c = bi.attn_qk_case(T=T, seed=8)
    kv = bi.kv_cache_case(T=T, seed=9)
    packed = torch.cat([c["q"].reshape(T, -1), c["k"].reshape(T, -1), kv["v"].reshape(T, -1)],
                       dim=1).to("cuda")
    q = packed[:, :48 * D].view(T, 48, D)
    k = packed[:, 48 * D:56 * D].view(T, 8, D)
    v = packed[:, 56 * D:].view(T, 8, D)
    got = run("ssmax", c, kv, True, q=q, k=k, v=v)
    check_caches("ssmax", c, kv, True, got, what="packed views")
    assert torch.equal(packed[:, 56 * D:].cpu(), kv["v"].reshape(T, -1))  # V is read only


def test_all_tokens_padding_writes_nothing():
    c = bi.attn_qk_case(T=40, seed=10)
    kv = bi.kv_cache_case(T=40, seed=11, pad_frac=1.0)
    q, k, gkc, gvc, init_k, init_v = run("rope", c, kv, False)
    assert np.array_equal(gkc, init_k) and np.array_equal(gvc, init_v)


def test_no_device_faults_after_cache_writes():
    torch.cuda.synchronize()
    assert rsn.beam_device_faults() == 0
