"""Multi-rank layout of the pass: the N blocks are independent, so ranks split them.

No collective touches the data path; ranks only agree on the timer (max over
ranks) and on which blocks each one owns.
"""
from __future__ import annotations


def block_range(n_total: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous blocks [lo, hi) owned by `rank` when n_total blocks are split over `world`."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(n_total, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def rank_seed(seed: int, rank: int) -> int:
    """Seed of a rank's own batch in weak scaling (every rank refines different blocks)."""
    return seed + 1000003 * rank


def max_over_ranks(value: float, device=None) -> float:
    """The slowest rank's value (the job's time); identity without a process group."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
