"""Replica bookkeeping for runs on N GPUs of one node.

The hot path has no exchange step on one GPU (each rank runs the whole
workload on its own device), so N-GPU runs are independent replicas; only the
timing is combined: every rank's time is reduced with MAX (the job ends when
the slowest rank ends) and the whole-job rate counts the work of all ranks.
"""
from __future__ import annotations

import os

import torch
import torch.distributed as dist


def rank_world() -> tuple[int, int, int]:
    """(rank, local_rank, world_size) from the launcher's environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")),
            int(os.environ.get("WORLD_SIZE", "1")))


def barrier() -> None:
    if dist.is_available() and dist.is_initialized() and dist.get_world_size() > 1:
        dist.barrier()


def max_over_ranks(x: float, device=None) -> float:
    """The maximum of x over all ranks (x itself on one rank)."""
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    if device is None:
        device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_rank: float, ms_max: float, world: int) -> float:
    """Work per second of the whole job: every rank's work over the slowest rank's time."""
    return world * work_per_rank / (ms_max * 1e-3)
