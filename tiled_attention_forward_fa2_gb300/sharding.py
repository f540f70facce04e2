"""Splitting a problem's (batch, head) slices over ranks.

Every (batch, head) slice of the attention forward is an independent problem
(its own Q, K, V rows and its own O, LSE rows), so a job spreads over GPUs by
giving each rank a contiguous block of the B*H slices: no data moves between
ranks and no collective is needed on the data path.  A contiguous block of the
[B, H, N, D] tensors is one contiguous byte range, so each rank calls the C ABI
with B = 1, H = its slice count and pointers offset to its block.
"""
from __future__ import annotations


def head_range(bh: int, rank: int, world: int) -> tuple[int, int]:
    """[start, stop) of the B*H slices rank ``rank`` of ``world`` computes: blocks
    whose sizes differ by at most one, in rank order, covering every slice once."""
    if world < 1 or not 0 <= rank < world or bh < 0:
        raise ValueError("need world >= 1, 0 <= rank < world, bh >= 0")
    return bh * rank // world, bh * (rank + 1) // world
