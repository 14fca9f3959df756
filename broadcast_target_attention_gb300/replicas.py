"""Data-parallel replicas: one process per GPU, each with its own batch.

IKBO target attention has no exchange step: the candidates of a batch, and
the batches themselves, are independent problems (each candidate reads only
its own user's K/V).  Running it on N GPUs therefore means N independent
replicas, each processing its own batch of the same shape, with no
collective on the data path.  The only collective is the host-side
reduction of the step time to its maximum over ranks (the job finishes when
the slowest rank does), so that whole-job throughput = the work all ranks
did / that time (weak scaling: work per GPU is fixed as N grows).
"""
from __future__ import annotations

import os
from dataclasses import replace
from typing import Tuple

from . import workloads as W

RANK_SEED_STRIDE = 1000


def dist_env() -> Tuple[int, int, int]:
    """(world_size, rank, local_rank) from the torchrun environment (1, 0, 0 without it)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def rank_config(name: str, rank: int) -> W.Config:
    """The batch of `rank`: the named workload with a seed of its own (rank 0 keeps the base seed)."""
    cfg = W.CONFIGS[name]
    return cfg if rank == 0 else replace(cfg, seed=cfg.seed + RANK_SEED_STRIDE * rank)


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a per-rank scalar over the default process group (x itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(work_per_rank: float, world_size: int, max_ms: float) -> float:
    """Whole-job rate: the work of all ranks over the slowest rank's time (per second)."""
    return work_per_rank * world_size / (max_ms * 1e-3)
