"""Host-side sharding of a frequency sweep over ranks (one GPU per rank).

Frequencies are independent (the sweep of malusrfworks.com, "Solving Dense
Matrices Fast in the Browser"), so a sweep shards by frequency with no
collective on the data path: each rank solves its own frequencies, and the
only exchange is the final gather of the solutions to rank 0.
"""
from __future__ import annotations

import numpy as np


def shard(nf: int, world: int, rank: int) -> np.ndarray:
    """Round-robin frequency indices owned by `rank` (every index exactly once)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    return np.arange(rank, nf, world, dtype=np.int64)


def max_over_ranks(value: float, device=None) -> float:
    """Max of a host scalar over all ranks (the timing rule for a multi-rank step)."""
    import torch
    import torch.distributed as dist

    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def gather_solutions(x_local: np.ndarray, nf: int, world: int, rank: int):
    """Assemble (nf, nrhs, n) solutions on rank 0 from each rank's shard (CPU arrays)."""
    import torch
    import torch.distributed as dist

    idx = shard(nf, world, rank)
    if world == 1:
        return x_local
    parts = [None] * world if rank == 0 else None
    dist.gather_object((idx, x_local), parts, dst=0)
    if rank != 0:
        return None
    shape = x_local.shape[1:]
    out = np.zeros((nf,) + shape, dtype=x_local.dtype)
    for ix, xs in parts:
        out[ix] = xs
    return out
