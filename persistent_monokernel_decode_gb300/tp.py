"""Tensor-parallel decode across GPUs: the partition of a decode layer and the reduction protocol (host side).

The monokernel pages run their 2B model with tensor parallelism over 8 GPUs and hide its collectives: a
custom collective layer keeps each exchange to a few microseconds inside the resident program, and "delayed
tensor parallelism" (creeta article, section "Delayed TP"; Kog blog, "Key technical innovations") moves the
reduction off the critical path so that it overlaps the next block's weight stream. Delayed TP proper needs a
model trained for it (the pages' Laneformer); for an ordinary Llama-style model the pages' fallback is the
overlap alone: a reduction runs while the next phase's weights keep streaming.

This library decodes on one GPU (the workloads fit in one GB300's HBM), so no multi-GPU kernel is built. This
module fixes what such a kernel would do, and is what the CPU tests exercise with two gloo processes:

* ``partition``: TP=W splits each layer Megatron-style. Rank r owns query heads [r Hq/W, (r+1) Hq/W) and the
  KV heads of those groups (Hkv % W == 0, so attention stays local), FFN rows [r F/W, (r+1) F/W) (gate and up
  rows of a pair stay together) and LM-head rows [r V/W, (r+1) V/W). Wo and Wd are split by columns, so their
  outputs are partial sums: two reductions per layer, plus a max-key reduction of the argmax per token.
* ``Mailbox`` / ``allreduce``: one exchange. Rank r writes its partial vector into slot r of every peer's
  mailbox (on GPUs: stores into the peer's HBM over NVLink, so the data lands in the reader's local memory
  before it is read), then publishes the exchange's sequence number in that slot's flag (a release store).
  Each rank waits for every peer's flag (acquire loads, bounded: a missing peer raises instead of hanging),
  then sums the W partials in rank order, so every rank gets bit-identical results. Mailboxes are
  double-buffered by the sequence number's parity: a rank can run at most one exchange ahead of the slowest
  peer (it needs every peer's partial to go on), so it never overwrites a slot a peer is still reading.
* Overlap: in the monokernel the consumer warps wait for the flags only when they stage the reduced vector
  for the next phase; the weight stream of that phase does not depend on it and keeps running.
"""
from __future__ import annotations

import time
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Shard:
    """What rank `rank` of a TP group of `world` owns in every layer (half-open ranges)."""
    world: int
    rank: int
    q_heads: tuple[int, int]
    kv_heads: tuple[int, int]
    ffn_rows: tuple[int, int]
    vocab_rows: tuple[int, int]


def partition(n_heads: int, n_kv_heads: int, ffn_dim: int, vocab: int, world: int, rank: int) -> Shard:
    """The TP=world shard of `rank`. Requires n_kv_heads, ffn_dim and vocab divisible by world (query-head
    groups, gate/up pairs and LM-head rows then split evenly)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank must be in [0, world)")
    if n_kv_heads % world or n_heads % n_kv_heads or ffn_dim % world or vocab % world:
        raise ValueError("n_kv_heads, ffn_dim and vocab must be multiples of the TP degree")
    g = n_heads // n_kv_heads

    def span(total):
        return (rank * total // world, (rank + 1) * total // world)

    kv = span(n_kv_heads)
    return Shard(world, rank, (kv[0] * g, kv[1] * g), kv, span(ffn_dim), span(vocab))


class ReductionTimeout(RuntimeError):
    """A peer's partial did not arrive within the wait limit."""


class Mailbox:
    """The receive side of one rank: for each sequence parity, W slots of n floats and W sequence flags.

    `buf` is a flat float64 view of memory every rank of the group can write (shared memory between the CPU
    test's processes; peer-mapped HBM on GPUs). Layout per rank: [2 parities][W flags] then [2][W][n] data.
    """

    def __init__(self, buf: np.ndarray, world: int, n: int, rank: int):
        self.world, self.n, self.rank = world, n, rank
        per_rank = Mailbox.floats_per_rank(world, n)
        if buf.size < world * per_rank:
            raise ValueError("mailbox buffer too small")
        self.buf = buf
        self.per_rank = per_rank

    @staticmethod
    def floats_per_rank(world: int, n: int) -> int:
        return 2 * world + 2 * world * n

    def _flag(self, owner: int, parity: int, slot: int) -> int:
        return owner * self.per_rank + parity * self.world + slot

    def _data(self, owner: int, parity: int, slot: int) -> slice:
        base = owner * self.per_rank + 2 * self.world + (parity * self.world + slot) * self.n
        return slice(base, base + self.n)

    def post(self, seq: int, partial: np.ndarray) -> None:
        """Write `partial` into slot `rank` of every peer's mailbox (and the own one), then its flag."""
        p = seq & 1
        for owner in range(self.world):
            self.buf[self._data(owner, p, self.rank)] = partial
        for owner in range(self.world):  # flags after all data: the release order of the device protocol
            self.buf[self._flag(owner, p, self.rank)] = float(seq)

    def take(self, seq: int, timeout_s: float) -> np.ndarray:
        """Wait (bounded) until every slot of exchange `seq` is in, then return their sum in rank order."""
        p = seq & 1
        t0 = time.monotonic()
        for slot in range(self.world):
            while self.buf[self._flag(self.rank, p, slot)] != float(seq):
                if time.monotonic() - t0 > timeout_s:
                    raise ReductionTimeout(f"rank {self.rank}: partial {seq} of rank {slot} did not arrive "
                                           f"within {timeout_s} s")
                time.sleep(1e-4)
        total = np.zeros(self.n, dtype=np.float32)
        for slot in range(self.world):  # fixed order: identical sums on every rank
            total = (total + self.buf[self._data(self.rank, p, slot)].astype(np.float32)).astype(np.float32)
        return total


def allreduce(mbox: Mailbox, seq: int, partial: np.ndarray, timeout_s: float = 5.0) -> np.ndarray:
    """Sum of every rank's `partial` (fp32, in rank order); `seq` numbers the exchanges of a launch from 1."""
    mbox.post(seq, np.asarray(partial, dtype=np.float32))
    return mbox.take(seq, timeout_s)


def argmax_key(value: float, index: int) -> int:
    """The 64-bit key whose maximum over ranks selects the largest logit, the lowest index among equal ones (the
    same ordering the single-GPU kernel folds with one atomicMax)."""
    u = int(np.float32(value).view(np.uint32))
    ordered = (~u & 0xFFFFFFFF) if (u & 0x80000000) else (u | 0x80000000)
    return (ordered << 32) | (0xFFFFFFFF - index)
