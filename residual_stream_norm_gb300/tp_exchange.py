"""Sequencing of the tensor-parallel partial exchange that feeds beam_allreduce_boundary_fwd.

Under tensor parallelism over P ranks every rank holds a partial sublayer output, and the fused
boundary on each rank needs all P partials, in rank order ("Serving Reflection Beam auf vLLM ab
Tag 0", "Agentengetriebene Optimierung", change 3: both TP all-reduces of a layer run inside the
norm kernel).  This module is the host-side protocol that hands each rank its peers' partials for
a step without a collective call:

  * Each rank's exchange buffer has `slots` slots; step s uses slot s % slots.
  * Rank r, at step s:
      1. waits until every rank has released slot s % slots from its previous use (step
         s - slots), so no partial is overwritten while a peer may still read it;
      2. writes its partial into that slot, then raises its ready flag for step s (the flag is
         written after the data: a reader that sees it sees the partial);
      3. waits until every rank's ready flag for step s is up, and reads the P partials of the
         slot in rank order (they go to beam_allreduce_boundary_fwd as x_parts[0..P-1]);
      4. raises its released flag for step s once the boundary no longer needs them.
  * Every wait is bounded: a peer that has not arrived within `timeout_s` raises
    ExchangeTimeout on the waiting rank, which can then leave between steps.

Every rank sums the same partials in the same order, so every rank computes bit-identical h'
and y, and the replicas of the residual stream cannot drift apart.

The transport carries the flags and the partials.  StoreTransport keeps both in a
torch.distributed Store (TCPStore or FileStore): the CPU stand-in that the gloo tests drive.  On
GPUs the partials would sit in device buffers that every peer has mapped, and the flags in
mapped words that each stream waits on before the boundary launch; that transport needs several
GPUs and is not part of this library.
"""
from __future__ import annotations

import datetime


class ExchangeTimeout(RuntimeError):
    """A peer did not raise its flag within the exchange's time limit."""


class StoreTransport:
    """Flags and partials in a torch.distributed Store: a flag is the presence of a key
    ``<kind>/<rank>/<step>``; rank r's partial for slot b is the value of ``part/<r>/<b>``."""

    def __init__(self, store, prefix: str = "tpx"):
        self.store = store
        self.prefix = prefix

    def _k(self, *parts) -> str:
        return "/".join([self.prefix, *map(str, parts)])

    def put(self, rank: int, slot: int, payload: bytes) -> None:
        self.store.set(self._k("part", rank, slot), payload)

    def get(self, rank: int, slot: int) -> bytes:
        return self.store.get(self._k("part", rank, slot))

    def raise_flag(self, kind: str, rank: int, step: int) -> None:
        self.store.set(self._k(kind, rank, step), b"1")

    def wait_flags(self, kind: str, ranks, step: int, timeout_s: float) -> None:
        keys = [self._k(kind, r, step) for r in ranks]
        try:
            self.store.wait(keys, datetime.timedelta(seconds=timeout_s))
        except Exception as e:  # the store's own timeout error
            missing = [r for r, k in zip(ranks, keys) if not self.store.check([k])]
            raise ExchangeTimeout(f"{kind} flag of step {step} missing from ranks {missing} "
                                  f"after {timeout_s} s") from e

    def drop_flags(self, kind: str, rank: int, step: int) -> None:
        try:
            self.store.delete_key(self._k(kind, rank, step))
        except Exception:
            pass


class PartialExchange:
    """The per-step protocol above for one rank.  publish(step, partial) then gather(step)
    returns the P partials in rank order; release(step) frees the slot for step + slots."""

    def __init__(self, transport, rank: int, world: int, timeout_s: float = 2.0,
                 slots: int = 2):
        if not 0 <= rank < world or slots < 1:
            raise ValueError("rank must be in [0, world) and slots >= 1")
        self.t, self.rank, self.world = transport, rank, world
        self.timeout_s, self.slots = timeout_s, slots
        self.ranks = list(range(world))

    def publish(self, step: int, partial: bytes) -> None:
        prev = step - self.slots
        if prev >= 0:  # every reader of this slot's previous contents is done with them
            self.t.wait_flags("released", self.ranks, prev, self.timeout_s)
        self.t.put(self.rank, step % self.slots, partial)
        self.t.raise_flag("ready", self.rank, step)
        old = step - 2 * self.slots  # no rank can still wait on flags this old
        if old >= 0:
            self.t.drop_flags("ready", self.rank, old)
            self.t.drop_flags("released", self.rank, old)

    def gather(self, step: int) -> list[bytes]:
        self.t.wait_flags("ready", self.ranks, step, self.timeout_s)
        return [self.t.get(r, step % self.slots) for r in self.ranks]

    def release(self, step: int) -> None:
        self.t.raise_flag("released", self.rank, step)
