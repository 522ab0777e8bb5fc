"""Rank sharding for running the path on several GPUs at once.

The fused op is independent per token row and the reduce-only op per
element, so G GPUs each take a contiguous block of rows (or elements) of the
global batch and exchange nothing: weak scaling with no data-path
collective.  The only cross-rank traffic is the timing barrier and the
max-over-ranks of the measured time.
"""
from __future__ import annotations


def shard_range(total: int, rank: int, world: int) -> tuple[int, int]:
    """[begin, end) of the contiguous block of `total` units owned by `rank`.

    Blocks differ in size by at most one unit and the first `total % world`
    ranks take the larger ones.
    """
    if world < 1 or not 0 <= rank < world or total < 0:
        raise ValueError(f"bad shard request: total={total} rank={rank} world={world}")
    base, extra = divmod(total, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks of the default process group (the value itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
