"""Replica helpers for N > 1 GPUs: requests are independent units, so every rank runs its own
model copy on its own requests; the only cross-rank steps are host-side bookkeeping (no
collective on the data path). One process per GPU, launched by torchrun."""
from __future__ import annotations

import os
from typing import List, Sequence, TypeVar

T = TypeVar("T")


def world() -> tuple:
    """(world_size, rank, local_rank) from the torchrun environment (1, 0, 0 without it)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard(units: Sequence[T], rank: int, world_size: int) -> List[T]:
    """Round-robin share of independent units (requests) for one rank."""
    if world_size < 1 or not 0 <= rank < world_size:
        raise ValueError("bad rank / world size")
    return [u for i, u in enumerate(units) if i % world_size == rank]


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of a per-rank timing over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())
