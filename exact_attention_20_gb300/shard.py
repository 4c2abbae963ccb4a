"""Host-side partitioning of independent attention problems across ranks.

The (batch, head) pairs of the forward pass are independent problems ("Each
block is independent of every other", section 2.8 of "Kernels and
FlashAttention: When the Same Math Runs 7.6x Faster"), so a job of B*H heads
splits across ranks with no exchange at all.  Splitting the keys of one head
instead needs one exchange step: each rank's normalised partial result is
merged through its logsumexp (the Flash-Decoding merge of "FlashAttention and
kernels.").  This module only computes index ranges; no attention arithmetic.
"""
from __future__ import annotations


def split_range(n: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous, balanced [start, stop) share of n units for `rank` of `world`.

    The first n % world ranks get one unit more; every unit is owned by
    exactly one rank, in order.
    """
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError("need world >= 1, 0 <= rank < world, n >= 0")
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return start, stop


def heads_for_rank(batch: int, heads: int, rank: int, world: int) -> list[tuple[int, int]]:
    """The (b, h) pairs rank `rank` owns, flattened b-major then h."""
    start, stop = split_range(batch * heads, rank, world)
    return [divmod(i, heads) for i in range(start, stop)]


def keys_for_rank(n_keys: int, rank: int, world: int) -> tuple[int, int]:
    """The key range [start, stop) rank `rank` attends over in a split-key run."""
    return split_range(n_keys, rank, world)
