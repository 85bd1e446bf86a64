"""Row sharding of one GEMM across ranks (one GPU each), with no data exchange.

C = A x B splits by rows of A and C with B replicated: rank r computes the
contiguous row block [lo, hi) of C from rows [lo, hi) of A.  Block edges are
multiples of the scheduled tile height (128, or 256 for CTA pairs), so every
output tile of a shard is an output tile of the unsharded plan and the shards,
put side by side, are bit for bit the unsharded result.  A K split would need
a reduction across ranks (the all-reduce of tensor-parallel row splits in the
H100 course notes, Lesson 10 "data/tensor parallelism"); it is not used.
"""
from __future__ import annotations


def m_shard(M: int, world: int, rank: int, align: int = 256):
    """Rows [lo, hi) of rank `rank` out of `world`: tile-aligned, as even as the alignment allows."""
    if world < 1 or not 0 <= rank < world or M < 0 or align < 1:
        raise ValueError("bad shard arguments")
    tiles = -(-M // align)
    t_lo = rank * tiles // world
    t_hi = (rank + 1) * tiles // world
    return min(M, t_lo * align), min(M, t_hi * align)
