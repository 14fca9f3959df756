"""The N > 1 path on CPU: two gloo ranks, as torchrun would start them.

One batch is sharded by user: each rank takes whole users with all their
candidates (longest first, balanced by candidates x keys) and computes their
rows from its shard alone; the union of the ranks' rows is the one-process
result.  The only collective is the max-over-ranks of the step time.  These
tests run that host logic with the oracle, and bench.py's reference arm under
torchrun, without a GPU.
"""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
BATCH = "ratio_1024x15"


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), OMP_NUM_THREADS="2")
    sys.path.insert(0, ROOT)
    import oracle
    from broadcast_target_attention_gb300 import partition as P
    from broadcast_target_attention_gb300 import workloads as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = P.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        full = W.generate(P.grown_config(BATCH, ws))
        users = P.assign_users(P.user_work(full.user_offsets, full.cand_to_user), ws)[r]
        sub, cands = P.shard(full, users)
        # this rank's rows, computed from its shard alone
        o = oracle.attention_wl(sub)
        # a per-rank "step time": the job ends with the slowest rank
        ms = P.max_over_ranks(1.0 + r)
        np.save(os.path.join(out_dir, f"out{r}.npy"), o)
        np.save(os.path.join(out_dir, f"cands{r}.npy"), cands)
        np.save(os.path.join(out_dir, f"users{r}.npy"), users)
        with open(os.path.join(out_dir, f"meta{r}.json"), "w") as f:
            json.dump({"ms": ms, "rate": P.job_throughput(full.n_cand, ms)}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_shard_one_batch_by_user(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    import oracle
    from broadcast_target_attention_gb300 import partition as P
    from broadcast_target_attention_gb300 import workloads as W
    full = W.generate(P.grown_config(BATCH, world))
    assert full.n_user == 2 * W.CONFIGS[BATCH].n_user and full.n_cand == 2 * W.CONFIGS[BATCH].n_cand
    meta = [json.load(open(tmp_path / f"meta{r}.json")) for r in range(world)]
    users = [np.load(tmp_path / f"users{r}.npy") for r in range(world)]
    # every user on exactly one rank
    assert sorted(np.concatenate(users).tolist()) == list(range(full.n_user))
    # the union of the ranks' rows, each row once, is the one-process result, bit for bit
    ref = oracle.attention_wl(full)
    out = np.full_like(ref, np.nan)
    seen = np.zeros(full.n_cand, dtype=np.int64)
    for r in range(world):
        cands = np.load(tmp_path / f"cands{r}.npy")
        P.scatter_rows(out, cands, np.load(tmp_path / f"out{r}.npy"))
        seen[cands] += 1
    assert np.all(seen == 1)
    np.testing.assert_array_equal(out, ref)
    # work balanced: the busier rank carries at most the mean plus the largest user
    work = P.user_work(full.user_offsets, full.cand_to_user)
    loads = [int(work[u].sum()) for u in users]
    assert max(loads) <= work.sum() / world + work.max()
    # every rank sees the same reduced time, the maximum; the rate counts the whole batch
    assert meta[0]["ms"] == meta[1]["ms"] == 2.0
    assert meta[0]["rate"] == pytest.approx(full.n_cand / 2e-3)


def test_assign_users_longest_first():
    from broadcast_target_attention_gb300 import partition as P
    work = np.array([5, 0, 9, 9, 1, 7, 3], dtype=np.int64)
    parts = P.assign_users(work, 3)
    # longest first, ties by index, to the least loaded rank (ties by rank):
    # 2 -> r0, 3 -> r1, 5 -> r2, 0 -> r2 (load 7 < 9), 6 -> r0 (9 = 9: lower rank),
    # 4 -> r1 (9 < 12), 1 -> r1 (10 < 12)
    assert [p.tolist() for p in parts] == [[2, 6], [1, 3, 4], [0, 5]]
    assert sorted(np.concatenate(parts).tolist()) == list(range(7))
    for ws in (1, 2, 3, 8):
        parts = P.assign_users(work, ws)
        loads = [int(work[p].sum()) for p in parts]
        assert max(loads) <= work.sum() / ws + work.max()
    # more ranks than users: some ranks get none
    parts = P.assign_users(np.array([4, 2]), 4)
    assert [len(p) for p in parts] == [1, 1, 0, 0]


def test_shard_keeps_each_users_rows_and_candidates():
    from broadcast_target_attention_gb300 import partition as P
    from broadcast_target_attention_gb300 import workloads as W
    wl = W.custom(n_user=5, counts=[3, 0, 2, 4, 1], lens=[7, 3, 0, 5, 9], H=2, D=64, Lq=2, seed=8,
                  shuffle=True)
    sub, cands = P.shard(wl, np.array([0, 3, 4]))
    off = wl.user_offsets.astype(np.int64)
    assert sub.user_offsets.tolist() == [0, 7, 12, 21]
    np.testing.assert_array_equal(sub.k[7:12], wl.k[off[3]:off[4]])
    np.testing.assert_array_equal(sub.v[12:21], wl.v[off[4]:off[5]])
    local = {0: 0, 3: 1, 4: 2}
    assert cands.tolist() == [c for c in range(wl.n_cand) if int(wl.cand_to_user[c]) in local]
    assert sub.cand_to_user.tolist() == [local[int(wl.cand_to_user[c])] for c in cands]
    np.testing.assert_array_equal(sub.q, wl.q[cands])
    # a user without candidates or keys is carried along harmlessly
    sub2, cands2 = P.shard(wl, np.array([1, 2]))
    assert sub2.n_cand == 2 and sub2.user_offsets.tolist() == [0, 3, 3]


def test_grown_config():
    from broadcast_target_attention_gb300 import partition as P
    from broadcast_target_attention_gb300 import workloads as W
    assert P.grown_config(BATCH, 1) is W.CONFIGS[BATCH]
    g = P.grown_config(BATCH, 4)
    assert (g.n_cand, g.n_user) == (4 * 1024, 4 * 15) and g.len_lo == W.CONFIGS[BATCH].len_lo
    with pytest.raises(ValueError):
        P.grown_config("tiny_8x2", 2)


def test_bench_reference_arm_under_torchrun():
    """Rank 0 alone runs the oracle arm and prints one JSON line; rank 1 exits 0."""
    env = dict(os.environ, OMP_NUM_THREADS="2")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr", "127.0.0.1", "--master-port", str(free_port()),
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--steps", "2", "--warmup", "3", "--config", "tiny_8x2"]
    p = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [json.loads(x) for x in p.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1
    line = lines[0]
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["cpu_baseline"]["kind"] == "oracle" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0
