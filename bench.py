"""Benchmark of the Beam sublayer-boundary path on GB300.

One step = one pass of every kernel of the path over an 8 x 2048 = 16384-token prefill batch
(hidden 5120, 48 query / 8 KV heads of 128, top-8 experts), all inputs resident in HBM:
    qk_norm_rope  ->  qk_norm_ssmax  ->  attn_gate  ->  boundary  ->  moe_combine_boundary
Every kernel streams more than the 129 MB L2 per launch, so no input survives in L2 from one
launch of it to the next.

Prints one JSON line (rank 0): whole-job tokens/s, per-kernel time / HBM GB/s / roofline
fraction, the roofline of the dominant kernel, the batch-1 decode chain (104 boundaries in one
CUDA graph, us per boundary), an end-to-end number through host buffers, the CPU oracle as a
baseline, and the SM clocks seen while the timed region ran.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Under torchrun each rank runs its own replica on its own GPU (the path has no exchange step):
the units are independent tokens, so N ranks process N batches ("weak" scaling).
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import beam_inputs as bi  # noqa: E402

METRIC = ("boundary tokens/s & HBM GB/s (% of GB300 peak) at T=16384; "
          "µs/boundary at T=1")
T_PREFILL = 16384
H = bi.HIDDEN
NQ, NKV, D, K = bi.N_Q_HEADS, bi.N_KV_HEADS, bi.HEAD_DIM, bi.TOP_K
FALLBACK_HBM_GBS = 6800.0

# Algorithmic HBM bytes per token of each kernel (reads + writes of the tensors it must touch).
BYTES_PER_TOKEN = {
    "qk_norm_rope": 2 * (NQ + NKV) * D * 2 + 8,       # Q, K read + written, position
    "qk_norm_ssmax": 2 * (NQ + NKV) * D * 2 + 8,
    "attn_gate": 3 * NQ * D * 2,                       # attn, gate read; out written
    "boundary": 4 * H * 2,                             # x, h read; h', y written
    "moe_combine_boundary": (K + 1) * H * 2 + 2 * H * 2 + K * 4,  # experts, h; h', y; weights
}
KERNELS = list(BYTES_PER_TOKEN)
# Rows beyond the five-kernel step, timed alone: the Q/K kernels fused with the KV-cache write
# (V read, slot read, K' and V rows written as FP8 E4M3, 1 byte per element).
KV_BYTES_PER_TOKEN = BYTES_PER_TOKEN["qk_norm_rope"] + NKV * D * 2 + 8 + 2 * NKV * D
# Grouped routing: 256 FP32 logits read, 8 int32 ids and 8 FP32 weights written.
ROUTE_BYTES_PER_TOKEN = bi.N_EXPERTS * 4 + K * 4 + K * 4
# The boundary with the tensor-parallel all-reduce fused ahead of it (TP8): the 8 partials and h
# read, h' and y written.
TP = bi.TP_RANKS
ALLREDUCE_BYTES_PER_TOKEN = (TP + 1) * H * 2 + 2 * H * 2
# Launches per kernel in the isolated timings (independent of --steps).
ISOLATED_LAUNCHES = 300
SOURCES = {
    "qk_norm_rope": "attention.cu", "qk_norm_ssmax": "attention.cu", "attn_gate": "attention.cu",
    "boundary": "boundary.cu", "moe_combine_boundary": "boundary.cu",
    "allreduce_boundary": "boundary.cu",
}


def bench_config(ws: int) -> dict:
    """The workload description both arms print (identical keys and values)."""
    return {"workload": "prefill 8x2048 = 16384 tokens at ~100K context: one pass of "
                        "qk_norm_rope, qk_norm_ssmax, attn_gate, boundary, "
                        "moe_combine_boundary (hidden 5120, 48/8 heads x 128, top-8)",
            "tokens_per_step": T_PREFILL, "hidden": H, "top_k": K,
            "l2": "inputs larger than L2 (every kernel streams >= 168 MB per launch; "
                  "L2 129 MB); no flush",
            "parallelism": f"replicas x{ws}"}


# ---------------------------------------------------------------------------------------------
# distributed plumbing
# ---------------------------------------------------------------------------------------------

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws: int, backend: str):
    if ws > 1 and not torch.distributed.is_initialized():
        torch.distributed.init_process_group(backend=backend)


def barrier(ws: int):
    if ws > 1:
        torch.distributed.barrier()


def whole_job_rate(ws: int, tokens_per_rank: int, steps: int, max_ms: float) -> float:
    """Tokens per second of the whole job: every rank processed its own batch each step, and the
    job took as long as its slowest rank."""
    return ws * tokens_per_rank * steps / (max_ms * 1e-3)


def max_over_ranks(x: float, ws: int, device) -> float:
    if ws == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) while the GPU is busy."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, device_index: int):
        self.rows = []
        self.proc = None
        self.ident = None
        try:
            uuid = torch.cuda.get_device_properties(device_index).uuid
            self.ident = f"GPU-{uuid}"
        except Exception:
            self.ident = None

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "100"]
        if self.ident:
            cmd += ["-i", self.ident]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except FileNotFoundError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) == 7:
                self.rows.append((time.perf_counter(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        rows = [r for t, r in self.rows if t0 - 0.15 <= t <= t1 + 0.15] or \
            [r for _, r in self.rows]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        reasons = sorted({self.REASONS[i] for r in rows for i in range(4)
                          if r[3 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows),
                "power_w_max": max((num(r[2]) or 0.0) for r in rows)}


# ---------------------------------------------------------------------------------------------
# workload
# ---------------------------------------------------------------------------------------------

def make_host_inputs(T: int, seed: int = 0) -> dict:
    """Seeded synthetic inputs of one step, on the host (pinned when CUDA is available)."""
    a_rope = bi.attn_qk_case(T=T, seed=seed, pos_mode="uniform")
    a_ss = bi.attn_qk_case(T=T, seed=seed + 1, pos_mode="contiguous")
    g = bi.gate_case(T=T, seed=seed + 2)
    pb = bi.prefill_boundary_case(T=T, seed=seed + 3)
    m = bi.moe_case(T=T, seed=seed + 4)
    host = {
        "q_r": a_rope["q"], "k_r": a_rope["k"], "pos_r": a_rope["pos"],
        "wq_r": a_rope["wq"], "wk_r": a_rope["wk"],
        "q_s": a_ss["q"], "k_s": a_ss["k"], "pos_s": a_ss["pos"],
        "wq_s": a_ss["wq"], "wk_s": a_ss["wk"],
        "attn": g["attn"], "gate": g["gate"], "bias": g["bias"],
        "h": pb["h"], "x": pb["x"], "w_post": pb["w_post"], "w_pre": pb["w_pre"],
        "h_m": m["h"], "e": m["e"], "topk_w": m["topk_w"],
        "w_post_m": m["w_post"], "w_pre_m": m["w_pre"],
    }
    if torch.cuda.is_available():
        host = {k: v.pin_memory() for k, v in host.items()}
    return host


INPUT_KEYS = ["q_r", "k_r", "pos_r", "q_s", "k_s", "pos_s", "attn", "gate", "bias", "h", "x",
              "h_m", "e", "topk_w"]
WEIGHT_KEYS = ["wq_r", "wk_r", "wq_s", "wk_s", "w_post", "w_pre", "w_post_m", "w_pre_m"]


class Step:
    """Device buffers of one step and the launch sequence through the C ABI."""

    def __init__(self, host: dict, device):
        import residual_stream_norm_gb300 as rsn
        self.rsn = rsn
        self.dev = {k: v.to(device, non_blocking=True) for k, v in host.items()}
        T = host["h"].shape[0]
        self.T = T
        d = self.dev
        self.out_gate = torch.empty_like(d["attn"])
        self.y = torch.empty_like(d["h"])
        self.y_m = torch.empty_like(d["h_m"])
        self.layer = 0
        self.lib = rsn.lib()

    def n_pair(self, i: int) -> tuple[int, int]:
        layer = i % 52
        return 2 * layer + 1, 2 * layer + 2

    def calls(self, i: int, st: int) -> tuple:
        """(entry point, arguments) of the five kernels of step i on the stream handle st."""
        d = self.dev
        n_attn, n_ffn = self.n_pair(i)
        wi = (n_attn - 1) % bi.N_BOUNDARIES
        return (
            ("beam_qk_norm_rope_fwd", (d["q_r"].data_ptr(), d["k_r"].data_ptr(), NQ * D, NKV * D,
                                        d["wq_r"].data_ptr(), d["wk_r"].data_ptr(),
                                        d["pos_r"].data_ptr(), self.T, NQ, NKV, D, bi.EPS,
                                        bi.ROPE_THETA, st)),
            ("beam_qk_norm_ssmax_fwd", (d["q_s"].data_ptr(), d["k_s"].data_ptr(), NQ * D, NKV * D,
                                         d["wq_s"].data_ptr(), d["wk_s"].data_ptr(),
                                         d["pos_s"].data_ptr(), self.T, NQ, NKV, D, bi.EPS,
                                         bi.SSMAX_BASE, bi.SSMAX_EXP, st)),
            ("beam_attn_gate_fwd", (self.out_gate.data_ptr(), d["attn"].data_ptr(),
                                     d["gate"].data_ptr(), d["bias"].data_ptr(), self.T, NQ, D,
                                     NQ * D, NQ * D, NQ * D, st)),
            ("beam_boundary_fwd", (d["h"].data_ptr(), self.y.data_ptr(), d["h"].data_ptr(),
                                    d["x"].data_ptr(), d["w_post"][wi].data_ptr(),
                                    d["w_pre"][wi].data_ptr(), self.T, H, n_attn, bi.EPS, None,
                                    st)),
            ("beam_moe_combine_boundary_fwd", (d["h_m"].data_ptr(), self.y_m.data_ptr(),
                                                d["h_m"].data_ptr(), d["e"].data_ptr(),
                                                d["topk_w"].data_ptr(), bi.ROUTED_SCALING,
                                                d["w_post_m"].data_ptr(), d["w_pre_m"].data_ptr(),
                                                self.T, H, K, n_ffn, bi.EPS, None, st)),
        )

    def launch(self, i: int, events=None) -> int:
        """Launch the five kernels of step i on the current stream; returns launches."""
        L, st = self.lib, torch.cuda.current_stream().cuda_stream
        rec = events.__getitem__ if events is not None else None
        calls = self.calls(i, st)
        for j, (fn, args) in enumerate(calls):
            if rec is not None:
                rec(j).record()
            stt = getattr(L, fn)(*args)
            if stt != 0:
                raise RuntimeError(f"{fn} returned {stt}")
        if rec is not None:
            rec(len(calls)).record()
        return len(calls)

    def kernel(self, j: int):
        """A closure that launches kernel j of step 0 alone on the current stream."""
        def run():
            fn, args = self.calls(0, torch.cuda.current_stream().cuda_stream)[j]
            stt = getattr(self.lib, fn)(*args)
            if stt != 0:
                raise RuntimeError(f"{fn} returned {stt}")
        return run

    def outputs(self):
        d = self.dev
        return [d["q_r"], d["k_r"], d["q_s"], d["k_s"], self.out_gate, d["h"], self.y, d["h_m"],
                self.y_m]


# ---------------------------------------------------------------------------------------------
# roofline inputs
# ---------------------------------------------------------------------------------------------

def measured_peak() -> tuple[float, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "of measured (MEASURED_PEAKS.json hbm_gbs, burst copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "of fallback (6.8 TB/s)"


def source_hash(name: str) -> str:
    """Digest of a kernel's source file and every header of the library (any change to them
    makes the committed DRAM counters stale)."""
    csrc = os.path.join(ROOT, "residual_stream_norm_gb300", "csrc")
    h = hashlib.sha256(open(os.path.join(csrc, SOURCES[name]), "rb").read())
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cuh", ".h")):
            h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def profiled_traffic(name: str, T: int):
    """DRAM bytes (read + write, read, write) per launch from the committed ncu capture, scaled to
    T tokens; None when the kernel source changed since the counters were taken."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)[name]
    except Exception:
        return None
    if rec.get("source_sha") != source_hash(name):
        return None
    per = T / float(rec["tokens_captured"])
    rd, wr = rec["dram_read_mb"] * 1e6 * per, rec["dram_write_mb"] * 1e6 * per
    return {"traffic": round(rd + wr, 1), "traffic_read": round(rd, 1),
            "traffic_write": round(wr, 1),
            "traffic_note": (f"ncu dram__bytes_read.sum / dram__bytes_write.sum of one launch at "
                             f"T={rec['tokens_captured']}, scaled to T={T}; reads match the "
                             "algorithmic input bytes, writes fall short by what is still dirty "
                             "in L2 when the kernel ends (not counted by the DRAM counters)")}


# ---------------------------------------------------------------------------------------------
# the oracle as CPU baseline
# ---------------------------------------------------------------------------------------------

def oracle_step(host: dict, lo: int, hi: int, i: int = 0):
    """The CPU oracle over tokens [lo, hi) of one step (all five operations)."""
    import oracle
    u = bi.u16
    n_attn, n_ffn = 2 * (i % 52) + 1, 2 * (i % 52) + 2
    wi = (n_attn - 1) % bi.N_BOUNDARIES
    s = slice(lo, hi)
    oracle.qk_norm_rope(u(host["q_r"][s]), u(host["k_r"][s]), u(host["wq_r"]), u(host["wk_r"]),
                        host["pos_r"][s].numpy())
    oracle.qk_norm_ssmax(u(host["q_s"][s]), u(host["k_s"][s]), u(host["wq_s"]), u(host["wk_s"]),
                         host["pos_s"][s].numpy())
    oracle.attn_gate(u(host["attn"][s]), u(host["gate"][s]), host["bias"].numpy(), NQ, D)
    oracle.boundary(u(host["h"][s]), u(host["x"][s]), u(host["w_post"][wi]), u(host["w_pre"][wi]),
                    n_attn)
    oracle.moe_combine_boundary(u(host["h_m"][s]), u(host["e"][s]), host["topk_w"][s].numpy(),
                                u(host["w_post_m"]), u(host["w_pre_m"]), n_ffn)


def time_oracle(host: dict, tokens: int, threads: int, i: int = 0) -> float:
    import oracle
    t0 = time.perf_counter()
    oracle.run_token_parallel(lambda lo, hi: oracle_step(host, lo, hi, i), tokens, threads)
    return time.perf_counter() - t0


# ---------------------------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------------------------

def copy_ceiling(device, nbytes: int = 1 << 30, reps: int = 20) -> dict:
    """A device-to-device copy of `nbytes` (well above L2) timed in this run: the bandwidth a
    plain stream of reads and writes reaches on this GPU right now, as a second ceiling beside
    the committed measured peak."""
    src = torch.empty(nbytes, dtype=torch.uint8, device=device)
    dst = torch.empty_like(src)
    src.fill_(1)
    for _ in range(3):
        dst.copy_(src)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record()
    for _ in range(reps):
        dst.copy_(src)
    e1.record()
    torch.cuda.synchronize(device)
    ms = e0.elapsed_time(e1) / reps
    del src, dst
    return {"gb_s": round(2 * nbytes / (ms * 1e-3) / 1e9, 1), "bytes_moved": 2 * nbytes,
            "how": "torch copy_ of a 1 GiB device buffer (read + write), 20 reps, CUDA events"}


def host_link(device, nbytes: int = 1 << 28, reps: int = 5, trials: int = 3) -> dict:
    """Pinned host <-> device copy bandwidth measured in this run: each direction alone, and both
    at once on two streams (the link's duplex capacity): the ceiling of the end-to-end number.
    The link is shared with the machine's other GPUs, so each figure is the best of `trials`
    timed rounds of `reps` copies, after an untimed round of the same pattern."""
    h = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d = torch.empty(nbytes, dtype=torch.uint8, device=device)
    h2 = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    d2 = torch.empty(nbytes, dtype=torch.uint8, device=device)
    s_in, s_out = torch.cuda.Stream(device), torch.cuda.Stream(device)
    cur = torch.cuda.current_stream(device)

    def timed(h2d: bool, d2h: bool) -> float:
        """GB/s of one round: `reps` copies in each enabled direction, each on its own stream."""
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        e0.record()
        for on, st, dst, src in ((h2d, s_in, d, h), (d2h, s_out, h2, d2)):
            if on:
                st.wait_event(e0)
                with torch.cuda.stream(st):
                    for _ in range(reps):
                        dst.copy_(src, non_blocking=True)
                cur.wait_stream(st)
        e1.record()
        torch.cuda.synchronize(device)
        return (int(h2d) + int(d2h)) * nbytes * reps / (e0.elapsed_time(e1) * 1e-3) / 1e9

    out = {}
    for name, dirs in (("h2d_gb_s", (True, False)), ("d2h_gb_s", (False, True)),
                       ("duplex_gb_s", (True, True))):
        timed(*dirs)  # untimed round of the same pattern
        out[name] = round(max(timed(*dirs) for _ in range(trials)), 1)
    del h, d, h2, d2
    return out


def decode_chain_us(device, replays: int = 200) -> dict:
    """Batch-1 decode: 104 boundary launches n = 1..104 captured in one CUDA graph."""
    import residual_stream_norm_gb300 as rsn
    ch = bi.decode_chain()
    h = ch["h0"].to(device)
    xs, wpo, wpr = ch["xs"].to(device), ch["w_post"].to(device), ch["w_pre"].to(device)
    y = torch.empty((bi.N_BOUNDARIES, 1, H), dtype=torch.bfloat16, device=device)
    L = rsn.lib()
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    g = torch.cuda.CUDAGraph()

    def chain(stream_handle):
        for i in range(bi.N_BOUNDARIES):
            st = L.beam_boundary_fwd(h.data_ptr(), y[i].data_ptr(), h.data_ptr(),
                                     xs[i].data_ptr(), wpo[i].data_ptr(), wpr[i].data_ptr(), 1, H,
                                     i + 1, bi.EPS, None, stream_handle)
            assert st == 0
    with torch.cuda.stream(s):
        chain(s.cuda_stream)  # warm
        with torch.cuda.graph(g, stream=s):
            chain(s.cuda_stream)
    torch.cuda.synchronize(device)
    for _ in range(10):
        g.replay()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    torch.cuda.synchronize(device)
    graph_us = e0.elapsed_time(e1) * 1e3 / replays / bi.N_BOUNDARIES
    # eager launches of the same chain (launch overhead included)
    e0.record()
    for _ in range(20):
        chain(torch.cuda.current_stream(device).cuda_stream)
    e1.record()
    torch.cuda.synchronize(device)
    eager_us = e0.elapsed_time(e1) * 1e3 / 20 / bi.N_BOUNDARIES
    return {"us_per_boundary": round(graph_us, 3), "boundaries": bi.N_BOUNDARIES,
            "graph_replays": replays, "eager_us_per_boundary": round(eager_us, 3),
            "T": 1, "note": "working set fits in L2: time only, no HBM GB/s"}


def time_isolated(fn, launches: int, device) -> float:
    """Mean ms per launch of `fn` over `launches` back-to-back launches on the current stream
    (after 5 warm-up launches), timed with CUDA events on that stream."""
    for _ in range(5):
        fn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(device)
    e0.record()
    for _ in range(launches):
        fn()
    e1.record()
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1) / launches


def graph_us(seq, replays: int, device) -> float:
    """Microseconds per replay of one CUDA graph that captures seq(stream_handle), warm; the
    launches inside are back to back with programmatic dependent launch."""
    s = torch.cuda.Stream(device)
    s.wait_stream(torch.cuda.current_stream(device))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        seq(s.cuda_stream)  # warm: first launches set up their kernels outside the capture
        with torch.cuda.graph(g, stream=s):
            seq(s.cuda_stream)
    torch.cuda.synchronize(device)
    for _ in range(10):
        g.replay()
    torch.cuda.synchronize(device)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(replays):
        g.replay()
    e1.record()
    torch.cuda.synchronize(device)
    return e0.elapsed_time(e1) * 1e3 / replays


def kernel_row(name: str, ms: float, by_per_token: int, T: int, peak: float) -> dict:
    by = by_per_token * T
    gbs = by / (ms * 1e-3) / 1e9
    return {"us": round(ms * 1e3, 2), "bytes_per_launch": by, "gb_s": round(gbs, 1),
            "frac_of_peak": round(gbs / peak, 4), "tokens_per_s": round(T / (ms * 1e-3), 1)}


def isolated_kernels(step: "Step", device, peak: float) -> dict:
    """Each kernel of the step timed alone over ISOLATED_LAUNCHES launches of its own at
    T = 16384 (inputs larger than L2, so no launch finds the previous one's data in L2)."""
    out = {}
    for j, name in enumerate(KERNELS):
        ms = time_isolated(step.kernel(j), ISOLATED_LAUNCHES, device)
        out[name] = kernel_row(name, ms, BYTES_PER_TOKEN[name], step.T, peak)
        out[name]["launches"] = ISOLATED_LAUNCHES
    return out


def allreduce_rows(device, peak: float) -> dict:
    """The boundary with the TP8 all-reduce fused ahead of it: T = 16384 (HBM roofline, the 8
    partials in this GPU's memory) timed alone, and the decode sizes T = 1 and T = 128 in CUDA
    graphs of 100 launches (L2-resident: time only)."""
    import residual_stream_norm_gb300 as rsn
    L = rsn.lib()
    out = {}
    c = bi.allreduce_case(T=T_PREFILL, P=TP, n=31, seed=11)
    h = c["h"].to(device)
    parts = c["parts"].to(device)
    del c
    y = torch.empty_like(h)
    ptrs = (ctypes.c_void_p * TP)(*[parts[p].data_ptr() for p in range(TP)])
    wpo = bi.norm_weight(bi.rng(12), H).to(device)
    wpr = bi.norm_weight(bi.rng(13), H).to(device)

    def launch(T, hh, yy, pp, st):
        stt = L.beam_allreduce_boundary_fwd(hh.data_ptr(), yy.data_ptr(), hh.data_ptr(), pp, TP,
                                            wpo.data_ptr(), wpr.data_ptr(), T, H, 31, bi.EPS,
                                            None, st)
        if stt != 0:
            raise RuntimeError(f"beam_allreduce_boundary_fwd returned {stt}")

    ms = time_isolated(lambda: launch(T_PREFILL, h, y, ptrs,
                                      torch.cuda.current_stream(device).cuda_stream),
                       ISOLATED_LAUNCHES, device)
    out["prefill_T16384_tp8"] = kernel_row("allreduce_boundary", ms, ALLREDUCE_BYTES_PER_TOKEN,
                                           T_PREFILL, peak)
    out["prefill_T16384_tp8"].update(launches=ISOLATED_LAUNCHES, partials=TP,
                                     bytes_per_token=ALLREDUCE_BYTES_PER_TOKEN)
    for T in (1, 128):
        hs, ys = h[:T].clone(), y[:T].clone()
        pt = (ctypes.c_void_p * TP)(*[parts[p, :T].data_ptr() for p in range(TP)])
        us = graph_us(lambda st: [launch(T, hs, ys, pt, st) for _ in range(100)], 50,
                      device) / 100
        out[f"decode_T{T}_tp8"] = {"us": round(us, 3), "tokens_per_s": round(T / (us * 1e-6), 1),
                                   "note": "CUDA graph of 100 launches; L2-resident: time only"}
    del parts
    return out


def small_configs(device) -> dict:
    """The workload's small configurations, each timed as CUDA graphs of back-to-back launches
    (warm; their working sets fit in L2, so time only, no HBM figure): the single boundary at
    T = 4; the 49 decode MoE boundaries (layers 3..51, own weights, T = 128) as one graph; the
    attention-side kernels at T = 128 and T = 2048."""
    import residual_stream_norm_gb300 as rsn
    L = rsn.lib()
    out = {}
    # config 1: single boundary, T = 4, n = 5
    c = bi.boundary_case(T=4, n=5, seed=0)
    h, x = c["h"].to(device), c["x"].to(device)
    y = torch.empty_like(h)
    wpo, wpr = c["w_post"].to(device), c["w_pre"].to(device)

    def b4(st):
        for _ in range(100):
            assert L.beam_boundary_fwd(h.data_ptr(), y.data_ptr(), h.data_ptr(), x.data_ptr(),
                                       wpo.data_ptr(), wpr.data_ptr(), 4, H, 5, bi.EPS, None,
                                       st) == 0
    us = graph_us(b4, 50, device) / 100
    out["1_single_boundary_T4"] = {"us": round(us, 3), "tokens_per_s": round(4 / (us * 1e-6), 1),
                                   "launches_per_graph": 100}
    # config 3: decode MoE boundary, T = 128, layers 3..51 in one graph
    m = bi.moe_case(T=128, seed=0)
    hm, e, w = m["h"].to(device), m["e"].to(device), m["topk_w"].to(device)
    ym = torch.empty_like(hm)
    g = bi.rng(99)
    layers = list(range(3, 52))
    ws = [(bi.norm_weight(g, H).to(device), bi.norm_weight(g, H).to(device)) for _ in layers]

    def moe49(st):
        for (wa, wb), layer in zip(ws, layers):
            assert L.beam_moe_combine_boundary_fwd(hm.data_ptr(), ym.data_ptr(), hm.data_ptr(),
                                                   e.data_ptr(), w.data_ptr(), bi.ROUTED_SCALING,
                                                   wa.data_ptr(), wb.data_ptr(), 128, H, K,
                                                   2 * layer + 2, bi.EPS, None, st) == 0
    us = graph_us(moe49, 50, device)
    out["3_decode_moe_T128_layers_3_51"] = {
        "us_per_launch": round(us / len(layers), 3), "us_per_49_launches": round(us, 2),
        "tokens_per_s": round(128 * len(layers) / (us * 1e-6), 1)}
    # config 4: attention side at T = 128 (positions U[0, 2^20)) and T = 2048 (contiguous)
    for T, mode in ((128, "uniform"), (2048, "contiguous")):
        a = bi.attn_qk_case(T=T, seed=T, pos_mode=mode)
        q, k = a["q"].to(device), a["k"].to(device)
        wq, wk, pos = a["wq"].to(device), a["wk"].to(device), a["pos"].to(device)
        gc = bi.gate_case(T=T, seed=T + 1)
        attn, gate, bias = gc["attn"].to(device), gc["gate"].to(device), gc["bias"].to(device)
        go = torch.empty_like(attn)
        row = {}
        for name in ("qk_norm_rope", "qk_norm_ssmax", "attn_gate"):
            def seq(st, name=name):
                for _ in range(50):
                    if name == "qk_norm_rope":
                        r = L.beam_qk_norm_rope_fwd(q.data_ptr(), k.data_ptr(), NQ * D, NKV * D,
                                                    wq.data_ptr(), wk.data_ptr(), pos.data_ptr(),
                                                    T, NQ, NKV, D, bi.EPS, bi.ROPE_THETA, st)
                    elif name == "qk_norm_ssmax":
                        r = L.beam_qk_norm_ssmax_fwd(q.data_ptr(), k.data_ptr(), NQ * D, NKV * D,
                                                     wq.data_ptr(), wk.data_ptr(),
                                                     pos.data_ptr(), T, NQ, NKV, D, bi.EPS,
                                                     bi.SSMAX_BASE, bi.SSMAX_EXP, st)
                    else:
                        r = L.beam_attn_gate_fwd(go.data_ptr(), attn.data_ptr(), gate.data_ptr(),
                                                 bias.data_ptr(), T, NQ, D, NQ * D, NQ * D,
                                                 NQ * D, st)
                    assert r == 0
            us = graph_us(seq, 20, device) / 50
            row[name] = {"us": round(us, 3), "tokens_per_s": round(T / (us * 1e-6), 1)}
        out[f"4_attention_T{T}"] = row
    out["note"] = "CUDA graphs of back-to-back launches, warm; L2-resident: time only"
    return out


def oracle_per_config(host: dict, threads: int) -> dict:
    """The oracle on each configuration of the workload, single-threaded and over token slices
    on all host cores (where the configuration has more than one token): ms per launch (per
    boundary for the decode chain) and tokens/s."""
    import oracle
    u = bi.u16

    def timed(fn, min_s=0.2):
        n, t0 = 0, time.perf_counter()
        while True:
            fn()
            n += 1
            el = time.perf_counter() - t0
            if el >= min_s:
                return el / n

    def both(call, T, sample=None):
        """call(lo, hi) over T tokens: single-threaded on `sample` tokens (scaled to T), and
        token-parallel over all of them."""
        ts = sample or T
        one = timed(lambda: call(0, ts)) * T / ts
        par = timed(lambda: oracle.run_token_parallel(call, T, threads)) if T > 1 else one
        used = min(threads, T)
        return {"ms_1core": round(one * 1e3, 3), "tokens_per_s_1core": round(T / one, 1),
                f"ms_{used}cores": round(par * 1e3, 3), "tokens_per_s_ncores": round(T / par, 1),
                "cores": used}

    out = {}
    c = bi.boundary_case(T=4, n=5, seed=0)
    hu, xu, wa, wb = u(c["h"]), u(c["x"]), u(c["w_post"]), u(c["w_pre"])
    out["1_single_boundary_T4"] = both(
        lambda lo, hi: oracle.boundary(hu[lo:hi], xu[lo:hi], wa, wb, 5), 4)
    ch = bi.decode_chain()
    h0, xs, wpo, wpr = u(ch["h0"]), u(ch["xs"]), u(ch["w_post"]), u(ch["w_pre"])

    def chain():
        hh = h0
        for i in range(bi.N_BOUNDARIES):
            hh, _, _ = oracle.boundary(hh, xs[i], wpo[i], wpr[i], i + 1)
    per = timed(chain) / bi.N_BOUNDARIES
    out["2_decode_chain_T1"] = {"ms_per_boundary_1core": round(per * 1e3, 4), "cores": 1,
                                "note": "one token: the chain is sequential"}
    m = bi.moe_case(T=128, seed=0)
    mh, me, mw, ma, mb = u(m["h"]), u(m["e"]), m["topk_w"].numpy(), u(m["w_post"]), u(m["w_pre"])
    out["3_decode_moe_T128"] = both(
        lambda lo, hi: oracle.moe_combine_boundary(mh[lo:hi], me[lo:hi], mw[lo:hi], ma, mb, 8),
        128)
    for T, mode in ((128, "uniform"), (2048, "contiguous")):
        a = bi.attn_qk_case(T=T, seed=T, pos_mode=mode)
        gc = bi.gate_case(T=T, seed=T + 1)
        aq, ak, awq, awk, ap = u(a["q"]), u(a["k"]), u(a["wq"]), u(a["wk"]), a["pos"].numpy()
        ga, gg, gb = u(gc["attn"]), u(gc["gate"]), gc["bias"].numpy()
        out[f"4_attention_T{T}"] = {
            "qk_norm_rope": both(lambda lo, hi: oracle.qk_norm_rope(aq[lo:hi], ak[lo:hi], awq,
                                                                     awk, ap[lo:hi]), T),
            "qk_norm_ssmax": both(lambda lo, hi: oracle.qk_norm_ssmax(aq[lo:hi], ak[lo:hi], awq,
                                                                       awk, ap[lo:hi]), T),
            "attn_gate": both(lambda lo, hi: oracle.attn_gate(ga[lo:hi], gg[lo:hi], gb, NQ, D),
                              T)}
    T = host["h"].shape[0]
    hh, xx = u(host["h"]), u(host["x"])
    w0, w1 = u(host["w_post"][0]), u(host["w_pre"][0])
    he, ee, ew = u(host["h_m"]), u(host["e"]), host["topk_w"].numpy()
    m0, m1 = u(host["w_post_m"]), u(host["w_pre_m"])
    out["5_prefill_T16384"] = {
        "boundary": both(lambda lo, hi: oracle.boundary(hh[lo:hi], xx[lo:hi], w0, w1, 1), T,
                         sample=1024),
        "moe_combine_boundary": both(
            lambda lo, hi: oracle.moe_combine_boundary(he[lo:hi], ee[lo:hi], ew[lo:hi], m0, m1,
                                                       2), T, sample=512),
        "note": "single-threaded figures from a sample of the first 1024 (512) tokens, scaled"}
    return out


def next_rows(host: dict, device, peak: float, iters: int = ISOLATED_LAUNCHES) -> dict:
    """Rows beyond the five-kernel step at the step's T, each launch timed alone with CUDA
    events: the Q/K kernels fused with an FP8 KV-cache write (inputs larger than L2), and the
    grouped routing (16.8 MB of logits: L2-resident between launches, so its GB/s is not an
    HBM figure; it is bound by the integer ALU work of its ranking)."""
    import residual_stream_norm_gb300 as rsn
    T = host["q_r"].shape[0]
    kv = bi.kv_cache_case(T=T, pad_frac=0.0, oob_frac=0.0, seed=7)
    d = {k: host[k].to(device) for k in ("q_r", "k_r", "pos_r", "wq_r", "wk_r", "q_s", "k_s",
                                         "pos_s", "wq_s", "wk_s")}
    v = kv["v"].to(device)
    slots = kv["slot_mapping"].to(device)
    kc = torch.zeros((kv["num_slots"], NKV, D), dtype=torch.uint8, device=device)
    vc = torch.zeros_like(kc)
    rc = bi.routing_case(T=T, seed=8)
    logits, rbias = rc["logits"].to(device), rc["bias"].to(device)
    rids = torch.empty((T, K), dtype=torch.int32, device=device)
    rw = torch.empty((T, K), dtype=torch.float32, device=device)
    runs = {
        "grouped_topk": lambda: rsn.beam_grouped_topk_fwd(rids, rw, logits, rbias),
        "qk_norm_rope_kv_fp8": lambda: rsn.beam_qk_norm_rope_kv_fwd(
            d["q_r"], d["k_r"], v, d["wq_r"], d["wk_r"], d["pos_r"], slots, kc, vc,
            cache_dtype=rsn.CACHE_FP8_E4M3),
        "qk_norm_ssmax_kv_fp8": lambda: rsn.beam_qk_norm_ssmax_kv_fwd(
            d["q_s"], d["k_s"], v, d["wq_s"], d["wk_s"], d["pos_s"], slots, kc, vc,
            cache_dtype=rsn.CACHE_FP8_E4M3),
    }
    out = {}
    for name, fn in runs.items():
        for _ in range(5):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(device)
        e0.record()
        for _ in range(iters):
            fn()
        e1.record()
        torch.cuda.synchronize(device)
        ms = e0.elapsed_time(e1) / iters
        by = (ROUTE_BYTES_PER_TOKEN if name == "grouped_topk" else KV_BYTES_PER_TOKEN) * T
        gbs = by / (ms * 1e-3) / 1e9
        out[name] = {"us": round(ms * 1e3, 2), "bytes_per_launch": by, "gb_s": round(gbs, 1),
                     "frac_of_peak": round(gbs / peak, 4),
                     "tokens_per_s": round(T / (ms * 1e-3), 1),
                     "launches": iters}
        if name != "grouped_topk":
            out[name]["cache"] = (f"FP8 E4M3, {kv['num_slots']} slots, one distinct random "
                                  "slot per token")
        else:
            out[name]["bound"] = "alu"
            out[name]["note"] = ("256 experts, 8 groups, top-4 groups, top-8; bound by the SM's "
                                 "integer ALU pipe (the ranking's compares and selects: 78% busy "
                                 "while the SMs are active, in the committed ncu capture), not "
                                 "by HBM; its GB/s fraction is not a roofline")
    return out


E2E_SETS = 3        # device buffer sets in flight
E2E_LANES = 2       # copy-in and copy-out streams each
E2E_TRIALS = 3      # pipelined runs; the line reports their median


def end_to_end(step: "Step", host: dict, device, ws: int, args) -> dict:
    """The step through host buffers: every step copies its inputs from pinned host memory,
    runs the five kernels through the C ABI and copies its results back to pinned host memory.
    Steps are pipelined the way a serving loop would run them: copy-in, compute and copy-out on
    their own streams over E2E_SETS device buffer sets, each copy direction spread over
    E2E_LANES streams (so that several copy engines can take part); events keep a buffer set
    from being refilled before its results have left.  The pipelined run is timed E2E_TRIALS
    times and the line reports the median, with every trial listed."""
    e2e_steps = max(2 * E2E_SETS, min(args.steps, 12))
    sets = [step] + [Step(host, device) for _ in range(E2E_SETS - 1)]
    outs = [st_.outputs() for st_ in sets]
    host_out = [torch.empty(o.shape, dtype=o.dtype, pin_memory=True) for o in outs[0]]
    h2d = sum(host[k].numel() * host[k].element_size() for k in INPUT_KEYS)
    d2h = sum(o.numel() * o.element_size() for o in outs[0])
    s_in = [torch.cuda.Stream(device) for _ in range(E2E_LANES)]
    s_out = [torch.cuda.Stream(device) for _ in range(E2E_LANES)]
    s_cmp = torch.cuda.Stream(device)
    ev_in = [[torch.cuda.Event() for _ in range(E2E_LANES)] for _ in range(E2E_SETS)]
    ev_out = [[torch.cuda.Event() for _ in range(E2E_LANES)] for _ in range(E2E_SETS)]
    ev_cmp = [torch.cuda.Event() for _ in range(E2E_SETS)]
    # inputs and outputs dealt to the lanes by size, largest first, to balance their bytes
    def deal(items):
        lanes, load = [[] for _ in range(E2E_LANES)], [0] * E2E_LANES
        for key, nbytes in sorted(items, key=lambda kv: -kv[1]):
            j = load.index(min(load))
            lanes[j].append(key)
            load[j] += nbytes
        return lanes
    in_lanes = deal([(k, host[k].numel() * host[k].element_size()) for k in INPUT_KEYS])
    out_lanes = deal([(j, o.numel() * o.element_size()) for j, o in enumerate(outs[0])])
    def trial() -> float:
        """ms of one pipelined run of e2e_steps steps (the slowest rank's)."""
        torch.cuda.synchronize(device)
        barrier(ws)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for s_ in s_in + s_out + [s_cmp]:
            s_.wait_event(e0)
        for i in range(e2e_steps):
            b = i % E2E_SETS
            for lane in range(E2E_LANES):
                st = s_in[lane]
                if i >= E2E_SETS:
                    for ev in ev_out[b]:
                        st.wait_event(ev)  # this set's previous results have left
                with torch.cuda.stream(st):
                    for k in in_lanes[lane]:
                        sets[b].dev[k].copy_(host[k], non_blocking=True)
                ev_in[b][lane].record(st)
            for ev in ev_in[b]:
                s_cmp.wait_event(ev)
            with torch.cuda.stream(s_cmp):
                sets[b].launch(i)
            ev_cmp[b].record(s_cmp)
            for lane in range(E2E_LANES):
                st = s_out[lane]
                st.wait_event(ev_cmp[b])
                with torch.cuda.stream(st):
                    for j in out_lanes[lane]:
                        host_out[j].copy_(outs[b][j], non_blocking=True)
                ev_out[b][lane].record(st)
        cur = torch.cuda.current_stream(device)
        for s_ in s_in + s_out + [s_cmp]:
            cur.wait_stream(s_)
        e1.record()
        torch.cuda.synchronize(device)
        return max_over_ranks(e0.elapsed_time(e1), ws, device)

    # The host link is shared with the machine's other GPUs: the median of E2E_TRIALS runs.
    trials = [trial() for _ in range(E2E_TRIALS)]
    e2e_ms = statistics.median(trials)
    T = step.T
    e2e = {"value": round(ws * T * e2e_steps / (e2e_ms * 1e-3), 1), "unit": "tokens/s",
           "trials": [round(ws * T * e2e_steps / (t * 1e-3), 1) for t in trials],
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "path": f"pinned host buffers -> cudaMemcpyAsync -> C ABI -> cudaMemcpyAsync -> host; "
                   f"copy-in ({E2E_LANES} streams), compute and copy-out ({E2E_LANES} streams) "
                   f"pipelined over {E2E_SETS} buffer sets; the host link bounds it (host_link: "
                   f"each direction's copy bandwidth measured in this run, and the bytes/s the "
                   f"pipelined run moved both ways)"}
    del sets[1:]
    e2e["host_link"] = host_link(device)
    e2e["host_link"]["e2e_gb_s"] = round((h2d + d2h) * e2e_steps / (e2e_ms * 1e-3) / 1e9, 1)
    e2e["host_link"]["e2e_frac_of_duplex"] = round(e2e["host_link"]["e2e_gb_s"] /
                                                   e2e["host_link"]["duplex_gb_s"], 3)
    return e2e


def run_gpu_arm(args) -> None:
    ws, rank, local = dist_env()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    init_dist(ws, "nccl")
    import residual_stream_norm_gb300 as rsn
    rsn.lib()  # fail loudly if the library is not built

    host = make_host_inputs(T_PREFILL, seed=rank)
    step = Step(host, device)
    torch.cuda.synchronize(device)

    nk = len(KERNELS)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)  # let the sampler come up before the warm-up steps (the GPU idles meanwhile)
    for i in range(args.warmup):
        step.launch(i)
    torch.cuda.synchronize(device)
    # The timed region: K steps, with events only at its two ends (nothing between the launches of
    # the step but the launches themselves).
    t0_ev, t1_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(ws)
    torch.cuda.synchronize(device)
    t_wall0 = time.perf_counter()
    t0_ev.record()
    gpu_launches = 0
    for i in range(args.steps):
        gpu_launches += step.launch(i)
    t1_ev.record()
    torch.cuda.synchronize(device)
    t_wall1 = time.perf_counter()
    barrier(ws)

    total_ms = t0_ev.elapsed_time(t1_ev)
    max_ms = max_over_ranks(total_ms, ws, device)
    T = step.T
    value = whole_job_rate(ws, T, args.steps, max_ms)

    # The same K steps again with an event between kernels: each kernel's time inside the step.
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    torch.cuda.synchronize(device)
    for i in range(args.steps):
        step.launch(i, events=ev[i])
    torch.cuda.synchronize(device)
    per_kernel_ms = {KERNELS[j]: sum(ev[i][j].elapsed_time(ev[i][j + 1]) for i in range(args.steps))
                     / args.steps for j in range(nk)}
    instrumented_ms = ev[0][0].elapsed_time(ev[-1][nk]) / args.steps

    peak, peak_src = measured_peak()
    # per kernel, in the step: the instrumented pass
    in_step = {}
    for name in KERNELS:
        in_step[name] = kernel_row(name, per_kernel_ms[name], BYTES_PER_TOKEN[name], T, peak)
        in_step[name]["share"] = round(per_kernel_ms[name] / sum(per_kernel_ms.values()), 4)
    dom = max(KERNELS, key=lambda k: per_kernel_ms[k])
    roofline = {"kernel": dom, "bound": "hbm", "achieved": in_step[dom]["gb_s"],
                "peak": peak, "unit": "GB/s", "frac": in_step[dom]["frac_of_peak"],
                "traffic": None, "peak_source": peak_src,
                "algorithmic_bytes_per_launch": in_step[dom]["bytes_per_launch"],
                "launches_timed": args.steps,
                "how": "algorithmic bytes / mean launch time of the kernel over the K steps run "
                       "again with a CUDA event between kernels (on the launching stream); "
                       "'isolated' is the kernel alone over back-to-back launches"}
    tr = profiled_traffic(dom, T)
    if tr:
        roofline.update(tr)

    # per kernel, alone: ISOLATED_LAUNCHES launches of its own (independent of --steps)
    t_iso0 = time.perf_counter()
    kernels = isolated_kernels(step, device, peak)
    for name in KERNELS:
        kernels[name]["share_in_step"] = in_step[name]["share"]
    roofline["isolated"] = {"us": kernels[dom]["us"], "gb_s": kernels[dom]["gb_s"],
                            "frac": kernels[dom]["frac_of_peak"],
                            "launches": ISOLATED_LAUNCHES}

    e2e = end_to_end(step, host, device, ws, args)
    decode = decode_chain_us(device)
    nxt = next_rows(host, device, peak)
    nxt["allreduce_boundary_tp8"] = allreduce_rows(device, peak)
    small = small_configs(device)
    t_iso1 = time.perf_counter()
    clocks.stop()
    ceiling = copy_ceiling(device)
    roofline["copy_ceiling_gbs"] = ceiling["gb_s"]
    roofline["frac_of_copy_ceiling"] = round(roofline["achieved"] / ceiling["gb_s"], 4)
    for v in kernels.values():
        v["frac_of_copy_ceiling"] = round(v["gb_s"] / ceiling["gb_s"], 4)

    out = None
    if rank == 0:
        threads = os.cpu_count() or 1
        cpu_s = time_oracle(host, T, threads)
        cpu = {"value": round(T / cpu_s, 1), "unit": "tokens/s", "cores": threads,
               "kind": "oracle",
               "sample": f"one full step ({T} tokens through all five operations), "
                         f"{threads} threads over token slices, {cpu_s:.2f} s wall",
               "per_config": oracle_per_config(host, threads)}
        b = kernels["boundary"]
        out = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(max_ms / args.steps, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage": "bf16",
            "data": "synthetic (seeded, Beam-shaped)",
            "config": bench_config(ws),
            "value_is": "tokens/s of the whole step (all five kernels over the same 16384 tokens), "
                        "timed with events at the ends of the K steps only",
            "ms_per_step_with_kernel_events": round(instrumented_ms, 4),
            "boundary_T16384": {"tokens_per_s": b["tokens_per_s"], "gb_s": b["gb_s"],
                                "frac_of_peak": b["frac_of_peak"], "us": b["us"],
                                "launches": ISOLATED_LAUNCHES},
            "decode_us_per_boundary": decode["us_per_boundary"],
            "kernels": kernels, "kernels_in_step": in_step, "roofline": roofline,
            "copy_ceiling": ceiling,
            "decode": decode, "configs": small, "next": nxt,
            "e2e": e2e,
            "cpu_baseline": cpu, "gpu_launches": gpu_launches * ws,
            "clocks": clocks.summary(t_wall0, t_wall1),
            "clocks_whole_run": clocks.summary(t_wall0, t_iso1),
            "wall_timed_s": round(t_wall1 - t_wall0, 4),
            "wall_isolated_s": round(t_iso1 - t_iso0, 2),
        }
    if ws > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    if out is not None:
        print(json.dumps(out), flush=True)


def run_reference_arm(args) -> None:
    """The CPU oracle, as it stands, timed on the host cores on the same workload."""
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    threads = os.cpu_count() or 1
    host = make_host_inputs(T_PREFILL, seed=0)
    T = T_PREFILL
    t_first = time_oracle(host, T, threads)
    # bound the run: at most ~150 s for warmup + steps
    per_step = max(64, min(T, int(T * 150.0 / max(1e-9, t_first * (args.steps + args.warmup)))))
    per_step -= per_step % 64
    for i in range(max(0, args.warmup - 1)):
        time_oracle(host, per_step, threads, i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        time_oracle(host, per_step, threads, i)
    el = time.perf_counter() - t0
    value = per_step * args.steps / el
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "storage": "bf16",
        "data": "synthetic (seeded, Beam-shaped)",
        "config": bench_config(ws),
        "cpu_baseline": {"value": round(value, 1), "unit": "tokens/s", "cores": threads,
                         "kind": "oracle",
                         "sample": f"{per_step} of the {T} tokens per step, all five operations"},
        "e2e": {"value": round(value, 1), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(out), flush=True)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    args = ap.parse_args(argv)
    if args.steps < 1:
        ap.error("--steps must be >= 1")
    if args.warmup < 3:
        # at least 3 untimed steps before the timed ones; the line reports the number done
        print(f"bench.py: --warmup {args.warmup} raised to 3", file=sys.stderr)
        args.warmup = 3
    if args.impl == "reference":
        run_reference_arm(args)
    else:
        run_gpu_arm(args)


if __name__ == "__main__":
    main()
