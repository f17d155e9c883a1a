"""GPU parity of the attention-side kernels against the CPU oracle (needs a GB300).

Per-head Q/K RMSNorm + RoPE (sliding-window layers) or + SSMax (NoPE layers), and the sigmoid
output gate ("Serving Reflection Beam auf vLLM ab Tag 0", section "Attention"; "SGLang 支撑编程模型
Beam 生产部署", "混合注意力与输出门控").  Decode (T = 128, positions U[0, 2^20)) and an 8 x 2048
prefill chunk at ~100K context (T = 2048, contiguous positions).
"""
import numpy as np
import pytest
import torch

import beam_inputs as bi
import oracle
import residual_stream_norm_gb300 as rsn
from tests._gpu import Guarded, dev, lib, u16
from tests._util import assert_bf16_close

pytestmark = pytest.mark.gpu
D = bi.HEAD_DIM


def run_qk(kind, c, q=None, k=None, **kw):
    q = dev(c["q"]) if q is None else q
    k = dev(c["k"]) if k is None else k
    fn = rsn.beam_qk_norm_rope_fwd if kind == "rope" else rsn.beam_qk_norm_ssmax_fwd
    fn(q, k, dev(c["wq"]), dev(c["wk"]), dev(c["pos"]), **kw)
    torch.cuda.synchronize()
    return q, k


def oracle_qk(kind, c, **kw):
    fn = oracle.qk_norm_rope if kind == "rope" else oracle.qk_norm_ssmax
    return fn(u16(c["q"]), u16(c["k"]), u16(c["wq"]), u16(c["wk"]), c["pos"].numpy(), **kw)


@pytest.mark.parametrize("kind", ["rope", "ssmax"])
@pytest.mark.parametrize("T,mode", [(128, "uniform"), (2048, "contiguous")])
def test_attention_side_config(kind, T, mode):
    lib()
    c = bi.attn_qk_case(T=T, seed=T, pos_mode=mode)
    q, k = run_qk(kind, c)
    wq, wk = oracle_qk(kind, c)
    assert_bf16_close(u16(q), wq, what=f"{kind} q T={T}")
    assert_bf16_close(u16(k), wk, what=f"{kind} k T={T}")


@pytest.mark.parametrize("kind", ["rope", "ssmax"])
@pytest.mark.parametrize("nq,nk", [(1, 0), (0, 1), (3, 2), (64, 8), (100, 3)])
def test_head_counts(kind, nq, nk):
    c = bi.attn_qk_case(T=5, n_q=nq, n_kv=nk, seed=nq * 10 + nk)
    q = dev(c["q"]) if nq else torch.empty((5, 0, D), dtype=torch.bfloat16, device="cuda")
    k = dev(c["k"]) if nk else torch.empty((5, 0, D), dtype=torch.bfloat16, device="cuda")
    q, k = run_qk(kind, c, q=q, k=k)
    wq, wk = oracle_qk(kind, c)
    assert_bf16_close(u16(q), wq, what=f"{kind} q {nq}/{nk}")
    assert_bf16_close(u16(k), wk, what=f"{kind} k {nq}/{nk}")


@pytest.mark.parametrize("kind", ["rope", "ssmax"])
@pytest.mark.parametrize("T,nq,nk", [(609, 48, 8), (1999, 48, 8), (1001, 3, 2), (1001, 1, 0),
                                     (1001, 0, 1), (1001, 64, 8), (4901, 48, 8), (4901, 3, 2),
                                     (4901, 1, 0), (4901, 64, 8)])
def test_many_tokens_ragged_tails(kind, T, nq, nk):
    # SSMax takes 4-token tiles from 4 tokens per SM on; RoPE one-token tiles up to 32 tokens per
    # SM and from there (4901 on a 152-SM GB300) the staged kernel's 8-token tiles, which copy the
    # next pass into shared memory: ragged last tiles and passes, and head counts whose items do
    # not fill a pass.
    c = bi.attn_qk_case(T=T, n_q=nq, n_kv=nk, seed=T + nq + nk)
    q = dev(c["q"]) if nq else torch.empty((T, 0, D), dtype=torch.bfloat16, device="cuda")
    k = dev(c["k"]) if nk else torch.empty((T, 0, D), dtype=torch.bfloat16, device="cuda")
    q, k = run_qk(kind, c, q=q, k=k)
    wq, wk = oracle_qk(kind, c)
    assert_bf16_close(u16(q), wq, what=f"{kind} q T={T} {nq}/{nk}")
    assert_bf16_close(u16(k), wk, what=f"{kind} k T={T} {nq}/{nk}")
    assert rsn.beam_device_faults() == 0


@pytest.mark.parametrize("kind", ["rope", "ssmax"])
@pytest.mark.parametrize("T", [37, 1001, 4901])
def test_views_into_packed_qkv_gate_projection(kind, T):
    # One packed [T, (48 + 8 + 8) * 128 + 48 * 128] projection output (Q | K | V | gate):
    # Q and K are row-strided views; V and the gate columns must stay untouched.
    c = bi.attn_qk_case(T=T, seed=21)
    g = bi.rng(22)
    v = bi.to_bf16(bi.normal(g, (T, 8 * D)))
    gate = bi.to_bf16(bi.normal(g, (T, 48 * D)))
    packed = torch.cat([c["q"].reshape(T, -1), c["k"].reshape(T, -1), v, gate], dim=1)
    buf = Guarded(tuple(packed.shape), fill=dev(packed))
    qv = buf.view[:, : 48 * D].view(T, 48, D)
    kv = buf.view[:, 48 * D: 56 * D].view(T, 8, D)
    run_qk(kind, c, q=qv, k=kv)
    buf.check()
    wq, wk = oracle_qk(kind, c)
    assert_bf16_close(u16(qv.contiguous()), wq, what="strided q")
    assert_bf16_close(u16(kv.contiguous()), wk, what="strided k")
    assert torch.equal(buf.view[:, 56 * D:].cpu(), torch.cat([v, gate], dim=1))


def test_rope_theta_and_special_positions():
    c = bi.attn_qk_case(T=8, seed=23)
    c["pos"] = torch.tensor([0, 1, 2, 511, 4095, 98_304, (1 << 20) - 1, (1 << 24) - 1],
                            dtype=torch.int64)
    for theta in (10000.0, 1e6):
        q, k = run_qk("rope", c, theta=theta)
        wq, wk = oracle_qk("rope", c, theta=theta)
        assert_bf16_close(u16(q), wq, what=f"rope theta={theta}")
        assert_bf16_close(u16(k), wk, what=f"rope theta={theta}")


@pytest.mark.parametrize("kind", ["rope", "ssmax"])
@pytest.mark.parametrize("T", [5, 1001, 4901])
def test_extreme_and_nonfinite_heads(kind, T):
    # Heads whose sum of squares sits near the top of the FP32 range, overflows, is NaN, is zero
    # or underflows; every other head random.  The kernels must give the oracle's IEEE results.
    c = bi.attn_qk_case(T=T, seed=61)
    q = u16(c["q"]).copy()
    def bits(v):  # BF16 bits of a value
        return int(oracle.bf16_rne(np.array([v], np.float32))[0])

    big = bits(1.3e19)                                # square 1.69e38: two of them stay finite
    for t in range(T):
        h = q[t]
        h[0, :] = 0
        h[0, 0] = h[0, 1] = big                       # one lane holds both large squares
        h[1, :] = 0
        h[1, 5] = bits(2e19)                          # its square overflows: the sum is inf
        h[2, 7] = 0x7FC0                              # NaN
        h[3, 9] = 0x7F80                              # +inf
        h[4, :] = 0                                   # all zero
        h[5, :] = bits(2.0 ** -70)                    # squares underflow
        h[6, 64] = big                                # partners of a large element
        h[6, 0] = bits(-1.3e19)
    c["q"] = bi.from_u16(q)
    qo, ko = run_qk(kind, c)
    wq, wk = oracle_qk(kind, c)
    assert_bf16_close(u16(qo), wq, what=f"{kind} extreme q T={T}")
    assert_bf16_close(u16(ko), wk, what=f"{kind} extreme k T={T}")


@pytest.mark.parametrize("kind", ["rope", "ssmax"])
@pytest.mark.parametrize("T", [5, 1001, 4901])
@pytest.mark.parametrize("eps", [0.0, 1e-2])
def test_eps_zero_and_large(kind, T, eps):
    # eps = 0: an all-zero head has r = 1/sqrt(0) = inf and NaN outputs, as in the oracle;
    # eps = 1e-2: the norm of small heads is dominated by eps
    c = bi.attn_qk_case(T=T, seed=71)
    q = u16(c["q"]).copy()
    q[:, 0, :] = 0
    small = (q[:, 1, :].astype(np.uint32) << 16).view(np.float32) * np.float32(2.0 ** -10)
    q[:, 1, :] = oracle.bf16_rne(small)
    c["q"] = bi.from_u16(q)
    qo, ko = run_qk(kind, c, eps=eps)
    wq, wk = oracle_qk(kind, c, eps=eps)
    assert_bf16_close(u16(qo), wq, what=f"{kind} eps={eps} q T={T}")
    assert_bf16_close(u16(ko), wk, what=f"{kind} eps={eps} k T={T}")


def test_ssmax_parameters_and_positions():
    c = bi.attn_qk_case(T=6, seed=24)
    c["pos"] = torch.tensor([0, 63487, 2095103, 7, 1 << 20, 123456], dtype=torch.int64)
    for base, ex in ((2048.0, 0.1), (512.0, 0.25)):
        q, k = run_qk("ssmax", c, ssmax_base=base, ssmax_exp=ex)
        wq, wk = oracle_qk("ssmax", c, base=base, expo=ex)
        assert_bf16_close(u16(q), wq, what=f"ssmax base={base}")
        assert_bf16_close(u16(k), wk, what=f"ssmax base={base}")


# ------------------------------------------------------------------------------------------
# gate
# ------------------------------------------------------------------------------------------

def run_gate(c, out=None, nh=bi.N_Q_HEADS, hd=D):
    attn = dev(c["attn"])
    out = torch.empty_like(attn) if out is None else out
    rsn.beam_attn_gate_fwd(out, attn, dev(c["gate"]), dev(c["bias"]), nh, hd)
    torch.cuda.synchronize()
    return out


def oracle_gate(c, nh=bi.N_Q_HEADS, hd=D):
    return oracle.attn_gate(u16(c["attn"]), u16(c["gate"]), c["bias"].numpy(), nh, hd)


@pytest.mark.parametrize("T", [128, 2048])
def test_gate_config(T):
    c = bi.gate_case(T=T, seed=T)
    assert_bf16_close(u16(run_gate(c)), oracle_gate(c), what=f"gate T={T}")


@pytest.mark.parametrize("nh,hd", [(1, 8), (3, 16), (5, 24), (48, 128), (7, 1024), (1024, 8),
                                   (1024, 1016)])
def test_gate_shapes(nh, hd):
    c = bi.gate_case(T=9, n_heads=nh, D=hd, seed=nh + hd)
    assert_bf16_close(u16(run_gate(c, nh=nh, hd=hd)), oracle_gate(c, nh, hd),
                      what=f"gate {nh}x{hd}")


def test_gate_switch_off_pass_through_and_in_place():
    c = bi.gate_case(T=17, seed=31)
    bias = c["bias"].clone()
    bias[0] = -float("inf")
    bias[1] = float("inf")
    c2 = dict(c, bias=bias)
    attn = dev(c["attn"])
    rsn.beam_attn_gate_fwd(attn, attn, dev(c["gate"]), dev(bias), bi.N_Q_HEADS, D)  # in place
    torch.cuda.synchronize()
    got = u16(attn)
    assert_bf16_close(got, oracle_gate(c2), what="gate in place")
    heads = got.reshape(17, bi.N_Q_HEADS, D)
    assert np.all((heads[:, 0] & 0x7FFF) == 0)                      # switched off
    assert np.array_equal(heads[:, 1], u16(c["attn"]).reshape(17, bi.N_Q_HEADS, D)[:, 1])


def test_gate_strided_rows_and_guards():
    T = 11
    c = bi.gate_case(T=T, seed=32)
    C = bi.N_Q_HEADS * D
    big = Guarded((T, C + 64), fill=dev(torch.cat([c["attn"], torch.zeros(T, 64,
                                                                         dtype=torch.bfloat16)],
                                                        dim=1)))
    gbuf = dev(torch.cat([c["gate"], torch.zeros(T, 128, dtype=torch.bfloat16)], dim=1))
    out = Guarded((T, C + 8))
    rsn.beam_attn_gate_fwd(out.view[:, :C], big.view[:, :C], gbuf[:, :C], dev(c["bias"]),
                           bi.N_Q_HEADS, D)
    torch.cuda.synchronize()
    big.check()
    out.check()
    assert_bf16_close(u16(out.view[:, :C].contiguous()), oracle_gate(c), what="strided gate")
    assert bool((out.view[:, C:] == -12345.0).all())


def test_zero_tokens():
    q = torch.empty((0, 48, D), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((0, 8, D), dtype=torch.bfloat16, device="cuda")
    w = torch.ones(D, dtype=torch.bfloat16, device="cuda")
    pos = torch.empty((0,), dtype=torch.int64, device="cuda")
    rsn.beam_qk_norm_rope_fwd(q, k, w, w, pos)
    rsn.beam_qk_norm_ssmax_fwd(q, k, w, w, pos)
    a = torch.empty((0, 48 * D), dtype=torch.bfloat16, device="cuda")
    rsn.beam_attn_gate_fwd(a, a, a, torch.zeros(48, device="cuda"), 48, D)
    torch.cuda.synchronize()


@pytest.mark.parametrize("kind", ["rope", "ssmax"])
@pytest.mark.parametrize("T", [3, 400, 1001])
def test_near_tie_head_sums(kind, T):
    # heads whose sum of squares sits at or just above an FP32 rounding boundary: the RoPE kernel
    # rounds its head sums exactly (its rotation can cancel), so its outputs are bit-identical;
    # the SSMax kernel sums in plain FP32 (its outputs only scale with r), within the parity bar
    c = bi.attn_qk_case(T=T, seed=41)
    g = np.random.Generator(np.random.PCG64(7))
    q = np.zeros((T, bi.N_Q_HEADS, D), np.float32)
    k = np.zeros((T, bi.N_KV_HEADS, D), np.float32)
    tiny = [0.0, 2.0 ** -30, 2.0 ** -40, 2.0 ** -60]
    for arr in (q, k):
        for idx in np.ndindex(arr.shape[:2]):
            cols = g.choice(D, size=3, replace=False)
            arr[idx][cols] = [1.0, 2.0 ** -12, tiny[(idx[0] + idx[1]) % 4]]
    c["q"] = bi.from_u16(oracle.bf16_rne(q))
    c["k"] = bi.from_u16(oracle.bf16_rne(k))
    qo, ko = run_qk(kind, c)
    wq, wk = oracle_qk(kind, c)
    if kind == "rope":
        assert np.array_equal(u16(qo), wq) and np.array_equal(u16(ko), wk)
    else:
        assert_bf16_close(u16(qo), wq, what=f"near-tie q T={T}")
        assert_bf16_close(u16(ko), wk, what=f"near-tie k T={T}")


def test_dependent_chain_across_kernels():
    # Programmatic dependent launch: each kernel may start before its predecessor finishes but
    # must read the predecessor's outputs only after it completes.  Chain RoPE -> gate (attn =
    # the rotated Q) -> boundary (x = the gated output) on one stream, back to back, twice (the
    # second pass reads the first's in-place results).  Each kernel is checked against the
    # oracle applied to the inputs it was given: the gate output, within the bar of the oracle's,
    # goes into the boundary as x, and through the cancelling sum bf16(a + b) a one-ulp
    # difference there may become several ulps of h', so the oracle's boundary takes the GPU's
    # gate output of each pass.
    T = 700
    a = bi.attn_qk_case(T=T, seed=51)
    g = bi.gate_case(T=T, seed=52)
    b = bi.boundary_case(T=T, H=bi.N_Q_HEADS * D, n=7, seed=53)
    q, k = dev(a["q"]), dev(a["k"])
    outs = [torch.empty((T, bi.N_Q_HEADS * D), dtype=torch.bfloat16, device="cuda")
            for _ in range(2)]
    ys = [torch.empty((T, bi.N_Q_HEADS * D), dtype=torch.bfloat16, device="cuda")
          for _ in range(2)]
    h = dev(b["h"])
    for p in range(2):
        rsn.beam_qk_norm_rope_fwd(q, k, dev(a["wq"]), dev(a["wk"]), dev(a["pos"]))
        rsn.beam_attn_gate_fwd(outs[p], q.view(T, -1), dev(g["gate"]), dev(g["bias"]),
                               bi.N_Q_HEADS)
        rsn.beam_boundary_fwd(h, ys[p], h, outs[p], dev(b["w_post"]), dev(b["w_pre"]), 7)
    torch.cuda.synchronize()
    oq, ok = u16(a["q"]), u16(a["k"])
    oh = u16(b["h"])
    for p in range(2):
        oq, ok = oracle.qk_norm_rope(oq, ok, u16(a["wq"]), u16(a["wk"]), a["pos"].numpy())
        og = oracle.attn_gate(oq.reshape(T, -1), u16(g["gate"]), g["bias"].numpy(), bi.N_Q_HEADS,
                              D)
        assert_bf16_close(u16(outs[p]), og, what=f"chain gate, pass {p}")
        oh, oy, _ = oracle.boundary(oh, u16(outs[p]), u16(b["w_post"]), u16(b["w_pre"]), 7)
        assert_bf16_close(u16(ys[p]), oy, what=f"chain y, pass {p}")
    assert_bf16_close(u16(q), oq, what="chain q")
    assert_bf16_close(u16(h), oh, what="chain h")

def _tie_heads(T, nh, seed, nudge_every=2):
    """Heads [T, nh, 128] whose sum of squares is an FP32 rounding midpoint exactly, or (every
    `nudge_every`-th head) lies just above one: four large elements +-a, one in each lane's
    vectors (vectors 0..3 belong to lanes 0..3 of the head's quad), so S0 = 4 a^2; small
    elements b, spread over all four lanes, adding exactly half an FP32 ulp of S0; and, for the
    nudged heads, a tiny t with t^2 ~ 2^-60 S0.  A plain or compensated FP32 sum rounds every one
    of them to S0; the exact sum rounds the nudged ones up.  a varies from head to head, so a sum
    taken from another quad, or one that misses a lane, moves r by far more than a BF16 ulp."""
    from fractions import Fraction
    g = np.random.Generator(np.random.PCG64(seed))
    x = np.zeros((T, nh, D), np.float64)
    t_i, h_i = np.meshgrid(np.arange(T), np.arange(nh), indexing="ij")
    m, e = (t_i * 7 + h_i * 3) % 8, (t_i + h_i) % 6 - 3
    a = (1 + m / 8) * 2.0 ** e                       # 4 significant bits: a^2 exact
    E = np.floor(np.log2(4 * a * a)).astype(np.int64)  # 4 a^2 in [2^E, 2^(E+1))
    even = E % 2 == 0
    b = np.where(even, 2.0 ** ((E - 28) // 2), 2.0 ** ((E - 27) // 2))  # 16 or 8 b^2 = 2^(E-24)
    nb = np.where(even, 16, 8)
    off = h_i % 8
    sign = lambda shape: np.where(g.random(shape) < 0.5, -1.0, 1.0)  # noqa: E731
    tt, hh = t_i.ravel(), h_i.ravel()
    for v in range(4):
        x[tt, hh, 8 * v + off.ravel()] = (a * sign(a.shape)).ravel()
    for i in range(16):
        sel = (nb > i).ravel()
        x[tt[sel], hh[sel], (8 * i + (off + 1) % 8).ravel()[sel]] = (b * sign(b.shape)).ravel()[sel]
    nudged = ((t_i * nh + h_i) % nudge_every == 0)
    tiny = 2.0 ** (E // 2 - 30)
    sel = nudged.ravel()
    x[tt[sel], hh[sel], (120 + (off + 2) % 8).ravel()[sel]] = tiny.ravel()[sel]
    # the construction, checked in exact rationals on a sample of heads: S = S0 + ulp(S0)/2
    # (+ t^2), an FP32 midpoint (or just above)
    for k in range(0, T * nh, max(1, T * nh // 200)):
        t, h = divmod(k, nh)
        ssum = sum(Fraction(float(v)) ** 2 for v in x[t, h] if v != 0)
        s0 = 4 * Fraction(float(a[t, h])) ** 2
        want = s0 + Fraction(2) ** int(E[t, h] - 24)
        if nudged[t, h]:
            want += Fraction(float(tiny[t, h])) ** 2
        assert ssum == want
    return oracle.bf16_rne(x.astype(np.float32))


@pytest.mark.parametrize("T,nq,nk", [(5, 48, 8), (5, 3, 2), (4, 5, 0), (3, 1, 1),
                                     (4 * 152 + 3, 48, 8), (4 * 152 + 3, 3, 2),
                                     (4 * 152 + 5, 1, 1), (32 * 152 + 3, 48, 8),
                                     (32 * 152 + 5, 3, 2)])
def test_near_tie_heads_in_every_quad_position(T, nq, nk):
    # RoPE head sums at an FP32 rounding midpoint, in every quad position of every warp, beside
    # inactive quads (head counts that leave a pass ragged: 3 + 2, 5 + 0, 1 + 1 heads, and a last
    # tile of 3 or 5 tokens) and, through the KV-cache kernel, beside V quads that take another
    # path.  Only the exact path rounds the nudged heads right, so the outputs are bit-identical
    # to the oracle only if that path runs, in every lane configuration, on its own quad's data.
    c = bi.attn_qk_case(T=T, n_q=nq, n_kv=nk, seed=T + nq + nk)
    c["q"] = bi.from_u16(_tie_heads(T, nq, seed=1)) if nq else c["q"]
    c["k"] = bi.from_u16(_tie_heads(T, nk, seed=2)) if nk else c["k"]
    wq, wk = oracle_qk("rope", c)
    q = dev(c["q"]) if nq else torch.empty((T, 0, D), dtype=torch.bfloat16, device="cuda")
    k = dev(c["k"]) if nk else torch.empty((T, 0, D), dtype=torch.bfloat16, device="cuda")
    qo, ko = run_qk("rope", c, q=q, k=k)
    assert np.array_equal(u16(qo), wq) and np.array_equal(u16(ko), wk), "rope"
    if nk == 0:
        return
    # the same heads through the KV-cache kernel (V quads interleaved with the norm quads)
    kv = bi.kv_cache_case(T=T, n_kv=nk, seed=T, pad_frac=0.1, oob_frac=0.05)
    q2 = dev(c["q"]) if nq else torch.empty((T, 0, D), dtype=torch.bfloat16, device="cuda")
    k2 = dev(c["k"])
    kc = torch.zeros((kv["num_slots"], nk, D), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    rsn.beam_qk_norm_rope_kv_fwd(q2, k2, dev(kv["v"]), dev(c["wq"]), dev(c["wk"]),
                                 dev(c["pos"]), dev(kv["slot_mapping"]), kc, vc)
    torch.cuda.synchronize()
    okc, ovc = oracle.kv_cache_write(np.zeros(kc.shape, np.uint16), np.zeros(vc.shape, np.uint16),
                                     wk, u16(kv["v"]), kv["slot_mapping"].numpy())
    assert np.array_equal(u16(q2), wq) and np.array_equal(u16(k2), wk), "rope + kv"
    assert np.array_equal(u16(kc), okc) and np.array_equal(u16(vc), ovc), "kv cache"
