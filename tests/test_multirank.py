"""The N > 1 path on CPU: two gloo ranks, as torchrun would start them.

Each rank processes its own batch (no exchange on the data path); the only
collective is the max-over-ranks of the step time.  These tests run that
host logic, and bench.py's reference arm under torchrun, without a GPU.
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


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import oracle
    from broadcast_target_attention_gb300 import replicas as R
    from broadcast_target_attention_gb300 import workloads as W

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = R.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        cfg = R.rank_config("tiny_8x2", r)
        wl = W.generate(cfg)
        # this rank's batch, computed with no help from the other rank
        o = oracle.attention_wl(wl)
        # a per-rank "step time": the job ends with the slowest rank
        ms = R.max_over_ranks(1.0 + r)
        np.save(os.path.join(out_dir, f"out{r}.npy"), o)
        with open(os.path.join(out_dir, f"meta{r}.json"), "w") as f:
            json.dump({"seed": cfg.seed, "ms": ms, "q0": float(wl.q.view(np.uint16)[0, 0, 0, 0]),
                       "rate": R.job_throughput(wl.n_cand, ws, ms)}, f)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_run_independent_batches(tmp_path):
    world = 2
    mp.start_processes(_rank_main, args=(world, free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    meta = [json.load(open(tmp_path / f"meta{r}.json")) for r in range(world)]
    outs = [np.load(tmp_path / f"out{r}.npy") for r in range(world)]
    # distinct seeds give distinct batches, rank 0 keeps the workload's own seed
    from broadcast_target_attention_gb300 import workloads as W
    assert meta[0]["seed"] == W.CONFIGS["tiny_8x2"].seed
    assert meta[0]["seed"] != meta[1]["seed"]
    assert not np.array_equal(outs[0], outs[1])
    # every rank sees the same reduced time: the maximum
    assert meta[0]["ms"] == meta[1]["ms"] == 2.0
    # whole-job rate: all ranks' candidates over the slowest rank's time
    assert meta[0]["rate"] == pytest.approx(2 * 8 / 2e-3)
    # a rank's result is the one-process result of that same batch
    import oracle
    from broadcast_target_attention_gb300 import replicas as R
    for r in range(world):
        ref = oracle.attention_wl(W.generate(R.rank_config("tiny_8x2", r)))
        np.testing.assert_array_equal(outs[r], ref)


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
