"""Multi-GPU runs: one process per GPU, each running its own replica of the
workload (the (batch, head) attention problems are independent, so there is
no collective on the data path). Only the timing is combined: the job time is
the slowest rank's, and the job throughput counts every rank's units.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def max_over_ranks(value: float, device=None) -> float:
    """Largest `value` over all ranks (the value itself when not distributed)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank: float, steps: int, job_ms: float, world: int) -> float:
    """Units per second of the whole job: every rank processed `units_per_rank`
    per step for `steps` steps, and the job took `job_ms` (max over ranks)."""
    return world * units_per_rank * steps / (job_ms / 1e3)
