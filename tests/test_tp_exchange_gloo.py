"""The tensor-parallel partial exchange on CPU ranks (gloo, 127.0.0.1; no GPU).

The host-side sequencing that hands every rank its peers' partial sublayer outputs for the fused
all-reduce boundary ("Serving Reflection Beam auf vLLM ab Tag 0", "Agentengetriebene
Optimierung", change 3): slots reused across steps, ready flags raised after the data, bounded
waits.  Each rank finishes the boundary with the oracle (the CPU stand-in for
beam_allreduce_boundary_fwd) on the partials it gathered; every rank must get the result of the
oracle on all partials in rank order, bit for bit, step after step.  A rank that stops
publishing makes its peers' next wait run out with ExchangeTimeout instead of hanging.
"""
import datetime
import hashlib
import os
import socket
import time

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import beam_inputs as bi
import oracle
from residual_stream_norm_gb300.tp_exchange import (ExchangeTimeout, PartialExchange,
                                                    StoreTransport)

T, H, STEPS = 3, 64, 6


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case(step: int, world: int):
    c = bi.allreduce_case(T=T, H=H, P=world, n=step + 1, seed=100 + step)
    if step == 1 and world >= 3:
        # rank order decides the result: (1, 2^-8, 2^-24, ...) rounds to 1 in rank order
        vals = [1.0, 2.0 ** -8] + [2.0 ** -24] * (world - 2)
        c["parts"] = torch.stack([torch.full((T, H), v, dtype=torch.bfloat16) for v in vals])
    return {k: (bi.u16(v) if isinstance(v, torch.Tensor) else v) for k, v in c.items()}


def _worker(rank: int, world: int, port: int, store_port: int, stop_at: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    store = dist.TCPStore("127.0.0.1", store_port, world, rank == 0,
                          timeout=datetime.timedelta(seconds=30))
    ex = PartialExchange(StoreTransport(store), rank, world, timeout_s=2.0, slots=2)
    digests, timed_out = [], None
    try:
        for step in range(STEPS):
            c = _case(step, world)
            if rank == world - 1 and step == stop_at:
                break  # this rank leaves between steps: it publishes nothing more
            ex.publish(step, c["parts"][rank].tobytes())
            t0 = time.perf_counter()
            try:
                got = ex.gather(step)
            except ExchangeTimeout:
                timed_out = (step, time.perf_counter() - t0)
                break
            parts = np.stack([np.frombuffer(b, np.uint16).reshape(T, H) for b in got])
            assert np.array_equal(parts, c["parts"]), "partials out of rank order"
            h_out, y, rstd = oracle.allreduce_boundary(c["h"], parts, c["w_post"], c["w_pre"],
                                                       c["n"])
            want = oracle.allreduce_boundary(c["h"], c["parts"], c["w_post"], c["w_pre"], c["n"])
            assert all(np.array_equal(a, b) for a, b in zip((h_out, y, rstd), want))
            ex.release(step)
            digests.append(hashlib.sha256(h_out.tobytes() + y.tobytes()).hexdigest())
        q.put((rank, digests, timed_out))
    finally:
        if stop_at >= STEPS:
            dist.barrier()
        dist.destroy_process_group()


def _run(world: int, stop_at: int = STEPS):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port, store_port = _free_port(), _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, store_port, stop_at, q))
             for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in range(world):
        r, d, to = q.get(timeout=180)
        out[r] = (d, to)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


@pytest.mark.parametrize("world", [2, 3])
def test_every_rank_gets_the_rank_order_result_step_after_step(world):
    out = _run(world)
    digests = [out[r][0] for r in range(world)]
    assert all(len(d) == STEPS for d in digests)
    assert all(d == digests[0] for d in digests), "ranks disagree"
    assert all(out[r][1] is None for r in range(world))


def test_a_rank_that_stops_publishing_times_its_peer_out():
    out = _run(2, stop_at=3)
    d0, to0 = out[0]
    assert len(d0) == 3                       # steps 0..2 completed
    assert to0 is not None and to0[0] == 3    # the wait of step 3 ran out
    assert 1.9 < to0[1] < 10.0                # after the 2 s limit, not a hang


def test_slot_reuse_waits_for_every_release():
    # one process, a FileStore: rank 0 cannot overwrite slot 0 (step 2) until both ranks have
    # released step 0
    import tempfile
    path = tempfile.mktemp()
    store = dist.FileStore(path, 2)
    a = PartialExchange(StoreTransport(store), 0, 2, timeout_s=0.5, slots=2)
    b = PartialExchange(StoreTransport(store), 1, 2, timeout_s=0.5, slots=2)
    for step in (0, 1):
        a.publish(step, b"a%d" % step)
        b.publish(step, b"b%d" % step)
        assert a.gather(step) == [b"a%d" % step, b"b%d" % step]
    a.release(0)
    with pytest.raises(ExchangeTimeout):
        a.publish(2, b"a2")                   # rank 1 has not released step 0
    b.release(0)
    a.publish(2, b"a2")
    assert a.t.get(0, 0) == b"a2" and b.gather(1) == [b"a1", b"b1"]
