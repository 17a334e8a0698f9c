"""Head split of the recurrence across ranks (one process per GPU).

The (sequence, head) chains of the recurrence are independent, so a problem
with H heads splits across `world` ranks by head with no collective on the
data path: rank r owns heads [lo, hi) of every tensor (q, k, v, g, beta, o
along the head axis, S along its head axis), runs the library on its slice,
and the full output is the concatenation of the ranks' slices along H.
"""
from __future__ import annotations


def head_range(H: int, world: int, rank: int) -> tuple[int, int]:
    """Heads [lo, hi) owned by `rank`: contiguous blocks, sizes differing by at most one."""
    if not 0 <= rank < world:
        raise ValueError("rank %d outside a world of %d" % (rank, world))
    base, extra = divmod(H, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def take_heads(x, lo: int, hi: int, axis: int):
    """The heads [lo, hi) of a tensor whose head axis is `axis`, made contiguous for the C ABI."""
    index = [slice(None)] * x.dim()
    index[axis] = slice(lo, hi)
    return x[tuple(index)].contiguous()
