"""Data-parallel partition of a parameter list into block-aligned shards.

Every 128-element block is parameter-local and every random draw is keyed by
the global element index, so a rank that owns a contiguous range of blocks of
a tensor steps it exactly as the whole tensor would be stepped, given the
shard's ``elem_offset``.  This module only computes the ranges (ZeRO-style:
the flattened parameter list cut into ``world`` nearly equal, block-aligned
pieces); it moves no data.

Factored parameters (rank >= 2 under the factored recipe) are the exception:
their row and column statistics span the whole parameter, so a shard of one
cannot be stepped on its own.  AReno docs "4-bit AdamW", section "State
representation": under data parallelism each rank's row and column sums of
g^2 are added over the group, and R and C are updated from the totals.  With the library that
is q4adamw_dp_factored_sums on every rank, a SUM all-reduce of the sums
buffers, then q4adamw_dp_step (include/q4adamw.h).  The buffers line up only
if every rank passes every factored parameter, in the same order, even where
it holds none of its elements: partition_all() gives that list.
"""
from __future__ import annotations

from dataclasses import dataclass

BLOCK = 128


@dataclass(frozen=True)
class Shard:
    tensor: int        # index in the parameter list
    start: int         # first element of the shard within the tensor (multiple of 128)
    numel: int         # elements in the shard

    @property
    def elem_offset(self) -> int:
        return self.start


def partition(numels, world: int, rank: int):
    """Shards of rank `rank` when the blocks of all tensors (in list order) are
    split into `world` contiguous runs of nearly equal block counts."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    nblocks = [(n + BLOCK - 1) // BLOCK for n in numels]
    total = sum(nblocks)
    lo = total * rank // world
    hi = total * (rank + 1) // world
    out = []
    base = 0
    for t, (n, nb) in enumerate(zip(numels, nblocks)):
        b0, b1 = max(lo, base), min(hi, base + nb)
        if b0 < b1:
            s = (b0 - base) * BLOCK
            e = min((b1 - base) * BLOCK, n)
            out.append(Shard(t, s, e - s))
        base += nb
    return out


def partition_all(numels, world: int, rank: int):
    """One shard per tensor, in list order: rank `rank`'s part as partition()
    gives it, or an empty shard (start 0, numel 0) where the rank holds none of
    the tensor -- the list a data-parallel factored step passes on every rank."""
    mine = {s.tensor: s for s in partition(numels, world, rank)}
    return [mine.get(t, Shard(t, 0, 0)) for t in range(len(numels))]
