"""GPU parity of beam_boundary_fwd against the CPU oracle (needs a GB300).

The boundary chain of "Serving Reflection Beam auf vLLM ab Tag 0" ("MoE und Residual-Stream";
"Agentengetriebene Optimierung", change 1) and "SGLang 支撑编程模型 Beam 生产部署"
("三明治归一化与深度缩放残差").  Bar: every BF16 output within 1 ulp of the oracle and at least
99.9 % bit-identical; the FP32 per-token scales within 2e-6 relative.
"""
import time

import numpy as np
import pytest
import torch

import beam_inputs as bi
import oracle
import residual_stream_norm_gb300 as rsn
from tests._gpu import CANARY, Guarded, dev, lib, persistent_T, u16
from tests._util import assert_bf16_close

pytestmark = pytest.mark.gpu

RSTD_RTOL = 2e-6


def run_gpu(h, x, w_post, w_pre, n, eps=bi.EPS):
    T, H = x.shape
    h_out = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(h_out)
    rstd = torch.empty((T, 2), dtype=torch.float32, device="cuda")
    rsn.beam_boundary_fwd(h_out, y, dev(h), dev(x), dev(w_post), dev(w_pre), n, eps, rstd)
    torch.cuda.synchronize()
    return u16(h_out), u16(y), rstd.cpu().numpy()


def check(got, want, what):
    (gh, gy, gr), (wh, wy, wr) = got, want
    assert_bf16_close(gh, wh, what=f"{what} h'")
    assert_bf16_close(gy, wy, what=f"{what} y")
    np.testing.assert_allclose(gr, wr, rtol=RSTD_RTOL, err_msg=f"{what} rstd")


def test_single_boundary_config():
    # T = 4 tokens, hidden 5120, n = 5, eps 1e-6, seed 0.
    lib()
    c = bi.boundary_case(T=4, n=5, seed=0)
    got = run_gpu(c["h"], c["x"], c["w_post"], c["w_pre"], 5)
    want = oracle.boundary(u16(c["h"]), u16(c["x"]), u16(c["w_post"]), u16(c["w_pre"]), 5)
    check(got, want, "T=4")


@pytest.mark.parametrize("T,H,n", [
    (1, 8, 1), (3, 16, 2), (2, 24, 3), (37, 5120, 7), (5, 5128, 104), (3, 16384, 11),
    (300, 5120, 9), (307, 4104, 50), (64, 16384, 1), (40, 5120, 1_000_000),
    # enough rows for the persistent TMA ring (>= 4 rows per SM), ragged and maximum H
    (700, 5120, 13), (613, 5128, 2), (1000, 16384, 104), (2000, 8, 3), (640, 24, 77),
    (650, 5120, 5000),
    # several rows per CTA through the row buffers, ragged rows
    (3001, 1032, 8), (1999, 5120, 21),
])
def test_shapes(T, H, n):
    c = bi.boundary_case(T=T, H=H, n=n, seed=T + H, outlier_frac=0.05, outlier_mult=16.0,
                         shared_scale=False)
    got = run_gpu(c["h"], c["x"], c["w_post"], c["w_pre"], n)
    want = oracle.boundary(u16(c["h"]), u16(c["x"]), u16(c["w_post"]), u16(c["w_pre"]), n)
    check(got, want, f"T={T} H={H} n={n}")


def test_decode_chain_104_boundaries():
    # Batch-1 decode: 104 successive boundaries n = 1..104, fresh x and own weights per
    # boundary; every pre-norm output and the final residual stream are compared.
    ch = bi.decode_chain()
    H = bi.HIDDEN
    h_gpu = dev(ch["h0"])
    xs, wpo, wpr = dev(ch["xs"]), dev(ch["w_post"]), dev(ch["w_pre"])
    y_gpu = torch.empty((bi.N_BOUNDARIES, 1, H), dtype=torch.bfloat16, device="cuda")
    for i in range(bi.N_BOUNDARIES):
        rsn.beam_boundary_fwd(h_gpu, y_gpu[i], h_gpu, xs[i], wpo[i], wpr[i], i + 1)
    torch.cuda.synchronize()
    h = u16(ch["h0"])
    xs_u, wpo_u, wpr_u = u16(ch["xs"]), u16(ch["w_post"]), u16(ch["w_pre"])
    ys = []
    for i in range(bi.N_BOUNDARIES):
        h, y, _ = oracle.boundary(h, xs_u[i], wpo_u[i], wpr_u[i], i + 1)
        ys.append(y)
    assert_bf16_close(u16(y_gpu), np.stack(ys), what="decode chain y_n")
    assert_bf16_close(u16(h_gpu), h, what="decode chain final h")


def test_decode_chain_in_cuda_graph_matches_eager():
    ch = bi.decode_chain(seed=3)
    H = bi.HIDDEN
    xs, wpo, wpr = dev(ch["xs"]), dev(ch["w_post"]), dev(ch["w_pre"])
    h_eager = dev(ch["h0"])
    y_eager = torch.empty((bi.N_BOUNDARIES, 1, H), dtype=torch.bfloat16, device="cuda")
    for i in range(bi.N_BOUNDARIES):
        rsn.beam_boundary_fwd(h_eager, y_eager[i], h_eager, xs[i], wpo[i], wpr[i], i + 1)
    h_graph = dev(ch["h0"])
    y_graph = torch.empty_like(y_eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(bi.N_BOUNDARIES):
                rsn.beam_boundary_fwd(h_graph, y_graph[i], h_graph, xs[i], wpo[i], wpr[i], i + 1)
    h_graph.copy_(dev(ch["h0"]))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(h_graph, h_eager) and torch.equal(y_graph, y_eager)


@pytest.mark.parametrize("n", [1, 2, 53, 104])
def test_prefill_16384_every_row(n):
    # 8 x 2048 prefill, full size, at the launch configuration the benchmark times; the oracle
    # recomputes every row (token slices on the host cores).
    c = bi.prefill_boundary_case()
    T = c["x"].shape[0]
    h, x = dev(c["h"]), dev(c["x"])
    wpo, wpr = dev(c["w_post"][n - 1]), dev(c["w_pre"][n - 1])
    h_out = torch.empty_like(h)
    y = torch.empty_like(h)
    rstd = torch.empty((T, 2), dtype=torch.float32, device="cuda")
    rsn.beam_boundary_fwd(h_out, y, h, x, wpo, wpr, n, bi.EPS, rstd)
    torch.cuda.synchronize()
    hu, xu = u16(c["h"]), u16(c["x"])
    wpo_u, wpr_u = u16(c["w_post"][n - 1]), u16(c["w_pre"][n - 1])
    parts = oracle.run_token_parallel(
        lambda lo, hi: oracle.boundary(hu[lo:hi], xu[lo:hi], wpo_u, wpr_u, n), T, 16)
    want = tuple(np.concatenate([p[i] for p in parts]) for i in range(3))
    check((u16(h_out), u16(y), rstd.cpu().numpy()), want, f"prefill n={n}")


@pytest.mark.parametrize("which,T,H", [
    ("rows", 33, 5120), ("rows", 33, 1032), ("rows", 33, 2056), ("rows", 33, 16384),
    ("rows", 320, 16384), ("persistent", 0, 5120)])
def test_in_place_aliasing(which, T, H):
    # h' over h and y over x, with guard bands; "persistent" takes T = 4 SMs + 5 rows, just enough
    # for the persistent prefetch kernel, whose row buffers are refilled while earlier rows of the
    # same buffers are written back.  The per-row kernel stores h' ahead of its second reduction;
    # the shapes give it 2, 1 (129 and 257 vectors: ragged warps), 4 and 8 vectors a thread
    T = T if which == "rows" else persistent_T()
    c = bi.boundary_case(T=T, H=H, n=6, seed=9)
    H = c["x"].shape[1]
    want = oracle.boundary(u16(c["h"]), u16(c["x"]), u16(c["w_post"]), u16(c["w_pre"]), 6)
    h, x = Guarded((T, H), fill=dev(c["h"])), Guarded((T, H), fill=dev(c["x"]))
    rsn.beam_boundary_fwd(h.view, x.view, h.view, x.view, dev(c["w_post"]), dev(c["w_pre"]), 6)
    torch.cuda.synchronize()
    h.check()
    x.check()
    assert_bf16_close(u16(h.view), want[0], what=f"in-place h' ({which}, T={T}, H={H})")
    assert_bf16_close(u16(x.view), want[1], what=f"in-place y ({which}, T={T}, H={H})")


def test_guard_bands_untouched():
    c = bi.boundary_case(T=19, H=5128, n=3, seed=10)
    T, H = c["x"].shape
    ho, yo = Guarded((T, H)), Guarded((T, H))
    rs = Guarded((T, 2), dtype=torch.float32)
    rsn.beam_boundary_fwd(ho.view, yo.view, dev(c["h"]), dev(c["x"]), dev(c["w_post"]),
                          dev(c["w_pre"]), 3, bi.EPS, rs.view)
    torch.cuda.synchronize()
    for g in (ho, yo, rs):
        g.check()
    want = oracle.boundary(u16(c["h"]), u16(c["x"]), u16(c["w_post"]), u16(c["w_pre"]), 3)
    check((u16(ho.view), u16(yo.view), rs.view.cpu().numpy()), want, "guarded")


def test_zero_tokens_is_a_no_op():
    h = torch.empty((0, 5120), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(5120, dtype=torch.bfloat16, device="cuda")
    rsn.beam_boundary_fwd(h, h, h, h, w, w, 3)
    out = Guarded((4, 5120))
    # a zero-token call on a view of a guarded buffer leaves everything as it was
    rsn.beam_boundary_fwd(out.view[:0], out.view[:0], out.view[:0], out.view[:0], w, w, 3)
    torch.cuda.synchronize()
    out.check()
    assert bool((out.view == -12345.0).all())


@pytest.mark.parametrize("T", [8, 700])
def test_nonfinite_and_degenerate_rows(T):
    # the first 8 rows degenerate (T = 700: the prefetch kernel), the rest random
    c = bi.boundary_case(T=T, n=4, seed=11)
    x = u16(c["x"]).copy()
    h = u16(c["h"]).copy()
    x[0, 17] = 0x7FC0          # NaN
    x[1, 3] = 0x7F80           # +inf
    x[2, :] = 0                # zero row: r = 1/sqrt(eps)
    x[3, :5] = 0x0001          # subnormals
    h[4, 100] = 0xFF80         # -inf in the residual
    x[5, :] = 0x7F7F           # largest finite: squares overflow FP32
    x[6, ::2] = 0x0080         # smallest normals
    x[7, :] = 0                # two squares of 1.69e38 in one thread: the row sum 3.38e38 is
    x[7, :2] = 0x5F34          # finite, though a partial sum seeded with the largest square is not
    hh, xx = bi.from_u16(h), bi.from_u16(x)
    got = run_gpu(hh, xx, c["w_post"], c["w_pre"], 4)
    want = oracle.boundary(h, x, u16(c["w_post"]), u16(c["w_pre"]), 4)
    assert_bf16_close(got[0], want[0], what="degenerate h'")
    assert_bf16_close(got[1], want[1], what="degenerate y")
    np.testing.assert_allclose(got[2], want[2], rtol=RSTD_RTOL)


def test_eps_zero_and_large():
    c = bi.boundary_case(T=6, n=2, seed=12)
    for eps in (0.0, 1e-2, 10.0):
        got = run_gpu(c["h"], c["x"], c["w_post"], c["w_pre"], 2, eps)
        want = oracle.boundary(u16(c["h"]), u16(c["x"]), u16(c["w_post"]), u16(c["w_pre"]), 2,
                               eps)
        check(got, want, f"eps={eps}")


def test_huge_weights_take_the_ieee_division_path():
    # |w_post| >= 2^120 can overflow x_hat to inf; those threads must divide by IEEE division.
    for T in (5, 700):
        c = bi.boundary_case(T=T, n=3, seed=12)
        w = u16(c["w_post"]).copy()
        w[::97] = 0x7E80  # 2^122
        w[5] = 0x7F7F     # largest finite BF16
        wb = bi.from_u16(w)
        got = run_gpu(c["h"], c["x"], wb, c["w_pre"], 3)
        want = oracle.boundary(u16(c["h"]), u16(c["x"]), w, u16(c["w_pre"]), 3)
        assert_bf16_close(got[0], want[0], what=f"huge w T={T} h'")
        assert_bf16_close(got[1], want[1], what=f"huge w T={T} y")


def test_no_device_faults_raised():
    # The persistent kernels bound every wait on their own copies; none may have given up.
    torch.cuda.synchronize()
    assert rsn.beam_device_faults() == 0


def _near_tie_rows(T, H, seed):
    """Rows whose sum of squares lies at or within 2^-60 relative of an FP32 rounding boundary
    (squares 1, 2^-24 and a tiny third term), so that only an exactly rounded sum gets r right."""
    g = np.random.Generator(np.random.PCG64(seed))
    x = np.zeros((T, H), np.float32)
    tiny = [0.0, 2.0 ** -30, 2.0 ** -40, 2.0 ** -60]
    for t in range(T):
        cols = g.choice(H, size=3, replace=False)
        base = [1.0, 1.0 + 2.0 ** -7][t % 2]          # even or odd FP32 neighbour below
        x[t, cols] = [base, 2.0 ** -12, tiny[t % 4] * (1 if g.random() < 0.5 else -1)]
    return oracle.bf16_rne(x)


@pytest.mark.parametrize("T", [7, 700])
def test_near_tie_row_sums_round_exactly(T):
    H = 5120
    xb = _near_tie_rows(T, H, seed=T)
    c = bi.boundary_case(T=T, n=3, seed=14)
    h = u16(c["h"])
    got = run_gpu(bi.from_u16(h), bi.from_u16(xb), c["w_post"], c["w_pre"], 3)
    want = oracle.boundary(h, xb, u16(c["w_post"]), u16(c["w_pre"]), 3)
    assert np.array_equal(got[2][:, 0], want[2][:, 0]), "r must be the exactly rounded value"
    check(got, want, f"near-tie rows T={T}")


def test_copy_timeout_path_sets_the_fault_word_and_leaves_the_context_usable():
    # A wait that nothing completes (an mbarrier armed for bytes no copy delivers) must give up
    # after its limit, raise the fault bit and return; the context then runs the next kernel.
    torch.cuda.synchronize()
    assert rsn.beam_device_faults(clear=True) == 0
    t0 = time.perf_counter()
    rsn.beam_selftest_copy_timeout(20_000_000)  # 20 ms
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert rsn.beam_device_faults(clear=True) == 1
    assert 0.015 < waited < 5.0
    c = bi.boundary_case(T=4, n=5, seed=0)
    got = run_gpu(c["h"], c["x"], c["w_post"], c["w_pre"], 5)
    want = oracle.boundary(u16(c["h"]), u16(c["x"]), u16(c["w_post"]), u16(c["w_pre"]), 5)
    check(got, want, "after the timeout")
    assert rsn.beam_device_faults() == 0


@pytest.mark.parametrize("kind", [0, 1])
def test_persistent_kernel_writes_nothing_once_its_wait_runs_out(kind):
    # The plain boundary's prefetch kernel (kind 0) and the MoE ring (kind 1), run with their
    # bulk copies withheld: every CTA's first wait on its own copies runs out after 20 ms.  No row
    # may reach h', y or rstd (the canaries stay, including an h that would be updated in place),
    # the fault bit is the signal, and the context runs the next launch correctly.  No fault,
    # trap or hang: the waits are the kernels' own bounded waits.
    torch.cuda.synchronize()
    assert rsn.beam_device_faults(clear=True) == 0
    T, H = persistent_T(), bi.HIDDEN
    ho, yo = Guarded((T, H), guard=256), Guarded((T, H), guard=256)
    rs = Guarded((T, 2), dtype=torch.float32, guard=256)
    g = bi.rng(kind)
    wpo, wpr = dev(bi.norm_weight(g, H)), dev(bi.norm_weight(g, H))
    t0 = time.perf_counter()
    rsn.beam_selftest_persistent_timeout(kind, ho.view, yo.view, wpo, wpr, limit_ns=20_000_000,
                                         rstd_out=rs.view)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert rsn.beam_device_faults(clear=True) == 1
    for buf in (ho, yo, rs):
        assert bool((buf.buf == CANARY).all()), "a row was written after the wait gave up"
    assert 0.015 < waited < 5.0
    c = bi.boundary_case(T=T, n=5, seed=0)
    got = run_gpu(c["h"], c["x"], c["w_post"], c["w_pre"], 5)
    want = oracle.boundary(u16(c["h"]), u16(c["x"]), u16(c["w_post"]), u16(c["w_pre"]), 5)
    check(got, want, "after the starved launch")
    assert rsn.beam_device_faults() == 0
