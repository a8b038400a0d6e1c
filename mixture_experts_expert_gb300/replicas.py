"""Timing across independent per-GPU replicas of the layer (weak scaling).

Each rank runs its own layer on its own GPU with no collective on the data path;
ranks only agree on the timing: the whole job took as long as its slowest rank, and
its throughput is the work of all ranks over that time.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def max_over_ranks(value: float, device: torch.device | str = "cpu") -> float:
    """The largest of every rank's ``value`` (the value itself on a single rank)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, world: int, seconds_slowest: float) -> float:
    """Units processed by all ranks per second of the slowest rank."""
    return units_per_rank * world / seconds_slowest
