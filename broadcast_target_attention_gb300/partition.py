"""One batch over several GPUs: users, with all their candidates, sharded across ranks.

IKBO target attention has no exchange step ("In-Kernel Broadcast Optimization",
§3.1: a candidate reads only its own user's keys and values), so the natural
shard of one batch is by user: rank r takes a set of whole users, their K/V
rows and every candidate of theirs, computes those candidates' rows alone, and
the union of the ranks' rows is the one-GPU result.  Users are dealt longest
first (largest r_u * L_u, candidates times keys: the work of a user) to the
rank with the least work so far, so the ranks' work is balanced.  There is no
collective on the data path; the only collective is the host-side maximum of
the step time (the job ends when the slowest rank does).  A gather is needed
only when one host tensor must hold all rows (`scatter_rows`).
"""
from __future__ import annotations

import os
from dataclasses import replace
from typing import List, Tuple

import numpy as np

from . import workloads as W


def dist_env() -> Tuple[int, int, int]:
    """(world_size, rank, local_rank) from the torchrun environment (1, 0, 0 without it)."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def user_work(user_offsets: np.ndarray, cand_to_user: np.ndarray) -> np.ndarray:
    """r_u * L_u for every user: its candidates times its keys (int64)."""
    off = np.asarray(user_offsets, dtype=np.int64)
    n_user = off.shape[0] - 1
    r = np.bincount(np.asarray(cand_to_user, dtype=np.int64), minlength=n_user)[:n_user]
    return r * np.diff(off)


def assign_users(work: np.ndarray, world_size: int) -> List[np.ndarray]:
    """Users of each rank, sorted by index: longest first (largest work, ties by index), each
    to the rank with the least work so far (ties by rank).  The busiest rank then carries at
    most the mean plus the largest single user's work."""
    work = np.asarray(work, dtype=np.int64)
    order = sorted(range(work.shape[0]), key=lambda u: (-int(work[u]), u))
    load = [0] * world_size
    mine: List[List[int]] = [[] for _ in range(world_size)]
    for u in order:
        r = min(range(world_size), key=lambda x: (load[x], x))
        mine[r].append(u)
        load[r] += int(work[u])
    return [np.asarray(sorted(m), dtype=np.int64) for m in mine]


def shard(wl: W.Workload, users: np.ndarray) -> Tuple[W.Workload, np.ndarray]:
    """The sub-batch of `users` (sorted): their K/V rows packed back to back in that order,
    their candidates in the batch's order with cand_to_user renumbered, and the batch
    indices of those candidates (where their rows go in the whole batch's output)."""
    users = np.asarray(users, dtype=np.int64)
    off = wl.user_offsets.astype(np.int64)
    lens = off[users + 1] - off[users]
    new_off = np.zeros(users.shape[0] + 1, dtype=np.int64)
    np.cumsum(lens, out=new_off[1:])
    rows = np.concatenate([np.arange(off[u], off[u + 1]) for u in users]) if users.size else \
        np.zeros(0, dtype=np.int64)
    local = np.full(wl.n_user, -1, dtype=np.int64)
    local[users] = np.arange(users.shape[0])
    c2u = wl.cand_to_user.astype(np.int64)
    cands = np.nonzero(local[c2u] >= 0)[0]
    cfg = replace(wl.cfg, name=f"{wl.cfg.name}[{users.shape[0]} users]", n_cand=int(cands.shape[0]),
                  n_user=int(users.shape[0]), counts=tuple(int(x) for x in np.bincount(
                      local[c2u[cands]], minlength=users.shape[0])) if users.size else (),
                  lens=tuple(int(x) for x in lens))
    sub = W.Workload(cfg=cfg, q=np.ascontiguousarray(wl.q[cands]), k=np.ascontiguousarray(wl.k[rows]),
                     v=np.ascontiguousarray(wl.v[rows]), user_offsets=new_off.astype(np.int32),
                     cand_to_user=local[c2u[cands]].astype(np.int32), scale=wl.scale)
    return sub, cands


def scatter_rows(out: np.ndarray, cands: np.ndarray, shard_rows: np.ndarray) -> None:
    """Put one rank's rows back at their candidates' places in the whole batch's output."""
    out[np.asarray(cands, dtype=np.int64)] = shard_rows


def grown_config(name: str, world_size: int) -> W.Config:
    """The batch that `world_size` GPUs share: the named workload with world_size times its
    users and candidates, drawn the same way (one batch, so per-GPU work stays that of
    the named workload as the GPUs grow).  world_size 1 gives the workload itself."""
    cfg = W.attention_config(name)
    if world_size == 1:
        return cfg
    if isinstance(cfg.counts, (tuple, list)) or isinstance(cfg.lens, (tuple, list)):
        raise ValueError(f"{name}: explicit per-user counts or lengths cannot be grown")
    return replace(cfg, name=f"{cfg.name}x{world_size}", n_cand=cfg.n_cand * world_size,
                   n_user=cfg.n_user * world_size,
                   forced_counts=tuple(cfg.forced_counts) * world_size)


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a per-rank scalar over the default process group (x itself without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(total_work: float, max_ms: float) -> float:
    """Whole-job rate: the work of all ranks over the slowest rank's time (per second)."""
    return total_work / (max_ms * 1e-3)
