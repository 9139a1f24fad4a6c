"""Counter ranges for fills split across processes (one per GPU).

A fill is a pure function of (seed, counter), and a fill cut at any element
equals the whole fill (tandem-sycl "Design", section Normals), so rank k of
W fills its own contiguous slice [offset, offset + length) of a global fill
by passing first_counter + offset: the ranks exchange nothing, and their
slices concatenated in rank order are the single-process fill.
"""
from __future__ import annotations


def shard(n_total: int, rank: int, world: int) -> tuple[int, int]:
    """(offset, length) of rank's slice of an n_total-element fill: the first
    n_total % world ranks take one element more than the others."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} is not in a world of {world}")
    if n_total < 0:
        raise ValueError("n_total must be non-negative")
    base, extra = divmod(n_total, world)
    length = base + (1 if rank < extra else 0)
    offset = rank * base + min(rank, extra)
    return offset, length


def first_counter(global_first: int, offset: int) -> int:
    """The first counter of a slice starting at element `offset` (mod 2^32)."""
    return (global_first + offset) & 0xFFFFFFFF
