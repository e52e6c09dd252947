"""Data-parallel partition of a parameter list into block-aligned shards.

Every 128-element block is parameter-local and every random draw is keyed by
the global element index, so a rank that owns a contiguous range of blocks of
a tensor steps it exactly as the whole tensor would be stepped, given the
shard's ``elem_offset``.  This module only computes the ranges (ZeRO-style:
the flattened parameter list cut into ``world`` nearly equal, block-aligned
pieces); it moves no data.
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
