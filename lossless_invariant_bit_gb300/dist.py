"""Multi-GPU plumbing for the IBP hot path: one process per GPU.

Every row decodes independently and the Mask/Bitval is a few KB, so the
path shards by partitioning the work -- an id batch (strong scaling) or the
stream of batches (weak scaling) -- with no collective on the data path.  The
only collectives are for measurement: a barrier around the timed region and
the maximum of the per-rank elapsed times.
"""
from __future__ import annotations

import os
from typing import Tuple


def rank_world() -> Tuple[int, int, int]:
    """(rank, local rank, world size) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def shard(n: int, rank: int, world: int) -> Tuple[int, int]:
    """Contiguous [start, start+count) share of n items for `rank`; the first
    n % world ranks take one extra item.  Shares tile [0, n) in rank order."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("rank %d outside world %d" % (rank, world))
    base, extra = divmod(int(n), world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def batch_seed(rank: int, batch: int) -> int:
    """Seed index of a rank's own id batch (weak scaling: disjoint per rank)."""
    return rank * 100_000 + batch


def max_over_ranks(value: float, dist, device=None) -> float:
    """Maximum of a float over all ranks (identity without a process group)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, dist, device=None) -> float:
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64,
                     device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())
