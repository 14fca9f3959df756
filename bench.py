"""Benchmark of IKBO target attention on GB300 -- prints ONE JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ikbo|reference]

A step is one pass of the whole hot path (the tcgen05 attention kernel, which
plans in-kernel for this batch) over one batch of the headline workload: 1024 candidates over 15
users (~70:1), user sequences of 256-1024 keys, H=4, D=128, Lq=1, bf16,
seeded synthetic inputs already resident in HBM.  L2 is flushed (a write
larger than L2) before every timed step.  The block of --steps timed steps is
repeated (`repeats` in the line) until it lasts --min-timed-s, so that the
clock samples come from inside the timed region; ms_per_step is the mean over
every timed step.  `value` is whole-job TFLOP/s
(4*H*D*Lq*S FLOPs, S = keys visited over all candidates); `e2e` is the same
metric through the host-buffer entry point with the copies inside the timed
region.  Under torchrun every rank runs its own replica (users shard with no
exchange); the time is the max over ranks.

--impl reference times the CPU fp64 oracle on the host cores on the same
workload (bounded samples), as the in-run baseline.

Other modes (one GPU each): --with-self (fused self + target attention),
--lce / --lce-ml (linear compression, two or three levels), --ml (attention
over a user -> vendor -> item hierarchy), --ratio-sweep (IKBO against the
explicit-broadcast path over candidate-to-user ratios).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from broadcast_target_attention_gb300 import accounting as A  # noqa: E402
from broadcast_target_attention_gb300 import partition as P  # noqa: E402
from broadcast_target_attention_gb300 import workloads as W  # noqa: E402

METRIC = "IKBO target-attn BF16 TFLOP/s & candidates/s (1024 cand/15 users); % of peak"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "source": "fallback"}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "source": "measured"}
    return dict(FALLBACK_PEAKS)


def workload_one_gpu(name: str):
    return W.generate(W.attention_config(name))


def config_block(wl, extra=None):
    c = wl.cfg
    d = {"workload": f"{c.name}: {c.description}", "n_cand": wl.n_cand, "n_user": wl.n_user,
         "H": c.H, "D": c.D, "Lq": c.Lq, "T_keys": wl.T, "S_keys_visited": wl.S,
         "l2": "flushed before every timed step (write of 2x L2 size)"}
    if extra:
        d.update(extra)
    return d


class ClockSampler:
    """SM clock and clock-event reasons while the GPU works, read (never set)
    through NVML by a poller process every ~1 ms; nvidia-smi sampling (every
    100 ms) when NVML cannot be loaded.  mark_start()/mark_end() bracket the
    timed region: the summary uses the samples inside it."""

    REASON_BITS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                   0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}
    SMI_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                  "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                  "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # In a process of its own, so that it samples whatever the benchmark's
    # Python thread is doing.  NVML clock type 1 is the SM clock.
    POLLER = r"""
import ctypes, sys, time
lib = ctypes.CDLL("libnvidia-ml.so.1")
assert lib.nvmlInit_v2() == 0
h = ctypes.c_void_p()
bus = sys.argv[1]
if not (bus and lib.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) == 0):
    assert lib.nvmlDeviceGetHandleByIndex_v2(int(sys.argv[2]), ctypes.byref(h)) == 0
reasons = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or lib.nvmlDeviceGetCurrentClocksThrottleReasons
clk, mx, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
print("ready", flush=True)
while True:
    if lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0 and lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
        r = rs.value if reasons(h, ctypes.byref(rs)) == 0 else 0
        print(time.monotonic(), clk.value, mx.value, r, flush=True)
    time.sleep(0.001)
"""

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []            # (t, sm_mhz, max_mhz, reason bits)
        self.window = [None, None]
        self.out = None
        self.proc = None
        self.path = None
        self.source = None

    def _start_nvml(self):
        import torch
        props = torch.cuda.get_device_properties(self.cuda_index)
        bus = ""
        if getattr(props, "pci_bus_id", None) is not None:
            bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id,
                                        getattr(props, "pci_device_id", 0))
        fd, self.path = tempfile.mkstemp(suffix=".txt")
        self.out = os.fdopen(fd, "w")
        self.proc = subprocess.Popen([sys.executable, "-c", self.POLLER, bus, str(self.cuda_index)],
                                     stdout=self.out, stderr=subprocess.DEVNULL)
        t_end = time.monotonic() + 10          # wait (bounded) until the poller runs
        while time.monotonic() < t_end and self.proc.poll() is None:
            with open(self.path) as f:
                if f.readline().startswith("ready"):
                    return
            time.sleep(0.01)
        raise RuntimeError("NVML poller did not start")

    def __enter__(self):
        try:
            self._start_nvml()
            self.source = "nvml"
        except Exception:
            if self.proc is not None:
                self.proc.kill()
                self.proc = None
            try:
                fd, self.path = tempfile.mkstemp(suffix=".csv")
                os.close(fd)
                self.proc = subprocess.Popen(
                    ["nvidia-smi", f"--id={self.cuda_index}", f"--query-gpu={self.SMI_FIELDS}",
                     "--format=csv,noheader,nounits", "-lms", "100", "-f", self.path],
                    stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
                self.source = "nvidia-smi"
            except Exception:
                self.proc = None
        return self

    def mark_start(self):
        self.window[0] = time.monotonic()

    def mark_end(self):
        self.window[1] = time.monotonic()

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.out is not None:
            self.out.close()

    def summary(self):
        if self.source == "nvml":
            with open(self.path) as f:
                for line in f:
                    parts = line.split()
                    if len(parts) == 4:
                        self.samples.append((float(parts[0]), float(parts[1]), float(parts[2]), int(parts[3])))
            os.unlink(self.path)
            t0, t1 = self.window
            inside = [x for x in self.samples if t0 is not None and t1 is not None and t0 <= x[0] <= t1]
            used = inside or self.samples
            if not used:
                return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "source": "nvml"}
            reasons = set()
            for x in used:
                for bit, name in self.REASON_BITS.items():
                    if x[3] & bit:
                        reasons.add(name)
            return {"sm_mhz": statistics.median(x[1] for x in used), "sm_max_mhz": max(x[2] for x in used),
                    "samples": len(used), "in_timed_region": bool(inside), "reasons": sorted(reasons),
                    "source": "nvml"}
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, val in zip(names, parts[5:9]):
                    if val.lower().startswith("active"):
                        reasons.add(n)
        os.unlink(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [x for x in sm if x > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons), "source": "nvidia-smi"}


# the files each tcgen05 attention kernel is compiled from
KERNEL_SOURCES = {
    "ikbo_attn_tc_kernel": ("ikbo_attn_tc.cuh", "ikbo_common.cuh", "ikbo_ptx.cuh"),
    "ikbo_attn_pp_kernel": ("ikbo_attn_pp.cuh", "ikbo_attn_tc.cuh", "ikbo_common.cuh", "ikbo_ptx.cuh"),
    "ikbo_attn_ab_kernel": ("ikbo_attn_ab.cuh", "ikbo_attn_tc.cuh", "ikbo_common.cuh", "ikbo_ptx.cuh"),
    "ikbo_lce_kernel": ("ikbo_lce.cuh", "ikbo_attn_tc.cuh", "ikbo_common.cuh", "ikbo_ptx.cuh"),
}


def lce_kernel_name(M: int, N: int) -> str:
    """The compression kernel a call of these sizes launches: CTA pairs (M = 256 MMAs) when M
    spans two to eight row tiles of 128 and N is 128 or 256, else one CTA per row tile."""
    mt = -(-M // 128)
    pairs = (N // 64) % 2 == 0 and 2 <= mt <= 8
    return f"ikbo_lce_kernel<{N // 64}, {'true' if pairs else 'false'}>"


def kernel_source_sha256(kernel_name: str = "ikbo_attn_tc_kernel") -> str:
    src = os.path.join(ROOT, "broadcast_target_attention_gb300", "csrc")
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES[kernel_name.split("<")[0]]:
        with open(os.path.join(src, fn), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def kernel_traffic(kernel_name: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(kernel_name, {}).get(workload)
    if not e:
        return None
    if e.get("source_sha256") != kernel_source_sha256(kernel_name):
        return None
    return float(e["dram_bytes_per_launch"])


def run_reference(args):
    """The oracle, as it stands, on the host cores: bounded samples of the workload."""
    ws, rank, _ = P.dist_env()
    if rank != 0:
        return
    import oracle
    wl = workload_one_gpu(args.config)
    c = wl.cfg
    L = np.diff(wl.user_offsets.astype(np.int64))
    cores = oracle.num_threads()
    # size each step's sample so the whole run stays within ~2 minutes
    t0 = time.perf_counter()
    probe = W.sample_candidates(wl, 64)
    oracle.attention_wl(wl, probe)
    per_cand = (time.perf_counter() - t0) / len(probe)
    budget_s = 120.0 / max(1, args.steps + args.warmup)
    n_sel = int(max(16, min(wl.n_cand, budget_s / max(per_cand, 1e-9))))
    sel = W.sample_candidates(wl, n_sel)
    flops = A.flops(c.H, c.D, c.Lq, int(L[wl.cand_to_user[sel]].sum()))
    for _ in range(args.warmup):
        oracle.attention_wl(wl, sel)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.attention_wl(wl, sel)
        times.append(time.perf_counter() - t0)
    t = statistics.mean(times)
    value = flops / t / 1e12
    sample = f"{len(sel)} of {wl.n_cand} candidates per step (all heads, all users represented)"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": t * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_block(wl, {"reference": "CPU fp64 oracle (broadcast, then softmax attention)"}),
        "candidates_per_s": len(sel) / t,
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(wl, seconds: float = 10.0):
    """The oracle timed on the host cores: whole-workload passes until ~`seconds` elapse."""
    import oracle
    c = wl.cfg
    cores = oracle.num_threads()
    sel = None
    L = np.diff(wl.user_offsets.astype(np.int64))
    t0 = time.perf_counter()
    probe = W.sample_candidates(wl, 64)
    oracle.attention_wl(wl, probe)
    per_cand = (time.perf_counter() - t0) / len(probe)
    if per_cand * wl.n_cand > seconds:
        sel = W.sample_candidates(wl, int(max(16, seconds / per_cand)))
    S = int(L[wl.cand_to_user[sel]].sum()) if sel is not None else wl.S
    flops = A.flops(c.H, c.D, c.Lq, S)
    runs, t_total = 0, 0.0
    while t_total < seconds and runs < 1000:
        t0 = time.perf_counter()
        oracle.attention_wl(wl, sel)
        t_total += time.perf_counter() - t0
        runs += 1
    n = wl.n_cand if sel is None else len(sel)
    return {"value": flops * runs / t_total / 1e12, "unit": "TFLOP/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{runs} passes over {n} of {wl.n_cand} candidates ({t_total:.1f} s of CPU work)"}


def run_ikbo(args):
    import torch
    import torch.distributed as dist

    import broadcast_target_attention_gb300 as ikbo

    ws, rank, local = P.dist_env()
    if ws > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ikbo.load()
    ikbo.set_kernel(args.kernel)
    # One batch for the whole job: the named workload grown N-fold for N ranks, its users
    # (with all their candidates) dealt to the ranks longest first; this rank runs its shard.
    full = W.generate(P.grown_config(args.config, ws))
    users = P.assign_users(P.user_work(full.user_offsets, full.cand_to_user), ws)[rank]
    wl = P.shard(full, users)[0] if ws > 1 else full
    c = full.cfg
    nums = A.workload_numbers(wl)
    flops, alg_bytes = nums["flops"], nums["alg_bytes"]
    total_flops = A.workload_numbers(full)["flops"]

    def t(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a)).view(dt).to(dev)

    q = t(wl.q.view(np.int16), torch.bfloat16)
    k = t(wl.k.view(np.int16), torch.bfloat16)
    v = t(wl.v.view(np.int16), torch.bfloat16)
    off = t(wl.user_offsets, torch.int32)
    c2u = t(wl.cand_to_user, torch.int32)
    out = torch.empty_like(q)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev)

    def step():
        ikbo.attn_fwd(q, k, v, off, c2u, wl.scale, out=out)

    def barrier():
        if ws > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            flush.fill_(1)
            step()
        assert ikbo.get_device_error() == 0
        # 1. timed steps: flush, then the hot path between two events, back to back.
        # The block of K steps is repeated R times, enqueued without a pause, so that the
        # timed region lasts long enough for the clock samples to fall inside it; R comes
        # from one untimed block and is the largest over the ranks.
        t0 = time.perf_counter()
        for i in range(args.steps):
            flush.fill_(i & 0xFF)
            step()
        barrier()
        block_s = max(time.perf_counter() - t0, 1e-6)
        repeats = P.max_over_ranks(float(max(1, int(np.ceil(args.min_timed_s / block_s)))), dev)
        repeats = int(min(repeats, max(1, 20000 // max(args.steps, 1))))
        n_timed = repeats * args.steps
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n_timed)]
        barrier()
        clk.mark_start()
        for i in range(n_timed):
            flush.fill_(i & 0xFF)
            starts[i].record()
            step()
            ends[i].record()
        barrier()
        clk.mark_end()
        step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
        # 1b. the same steps with no flush between them (inputs L2-resident), for reference.
        # A GPU-side pause (touching no memory) before each keeps the host's enqueue ahead
        # of the GPU, so that no step's events take in the host's launch time.
        for i in range(min(args.steps, 200)):
            torch.cuda._sleep(100_000)
            starts[i].record()
            step()
            ends[i].record()
        torch.cuda.synchronize(dev)
        hot = [starts[i].elapsed_time(ends[i]) for i in range(min(args.steps, 200))]
        # 2. per-kernel durations (events recorded by the library around each kernel)
        ikbo.set_timing(True)
        plan_ms, attn_ms = [], []
        for i in range(min(args.steps, 200)):
            flush.fill_(i & 0xFF)
            step()
            a, b = ikbo.get_timing()
            plan_ms.append(a)
            attn_ms.append(b)
        ikbo.set_timing(False)
        # 3. end to end through the host-buffer entry point
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        hoff, hc2u = off.cpu().pin_memory(), c2u.cpu().pin_memory()
        hout = torch.empty_like(hq).pin_memory()
        for _ in range(3):
            ikbo.attn_fwd_host(hq, hk, hv, hoff, hc2u, wl.scale, out=hout)
        e2e_ms = []
        n_e2e = min(args.steps, 50)
        for _ in range(n_e2e):
            t0 = time.perf_counter()
            ikbo.attn_fwd_host(hq, hk, hv, hoff, hc2u, wl.scale, out=hout)
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
        # 4. the explicit-broadcast comparison path
        bout = torch.empty_like(q)
        ikbo.broadcast_attn_fwd(q, k, v, off, c2u, wl.scale, out=bout)
        ikbo.set_timing(True)
        bc_ms = []
        for i in range(min(args.steps, 20)):
            flush.fill_(i & 0xFF)
            ikbo.broadcast_attn_fwd(q, k, v, off, c2u, wl.scale, out=bout)
            bc_ms.append(ikbo.get_timing()[1])
        ikbo.set_timing(False)
    assert ikbo.get_device_error() == 0
    clocks = clk.summary()

    ms = P.max_over_ranks(statistics.mean(step_ms), dev)
    value = P.job_throughput(total_flops, ms) / 1e12
    pk = peaks()
    attn = statistics.mean(attn_ms)
    achieved_gbs = alg_bytes / (attn * 1e-3) / 1e9
    kname = f"{ikbo.KERNEL_NAMES[ikbo.selected_kernel(wl.n_cand, wl.n_user, c.H, c.Lq, c.D)]}<{c.D}>"
    traffic = kernel_traffic(kname, c.name)
    ai = flops / alg_bytes
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if ai < ridge:
        roof = {"bound": "hbm", "achieved": achieved_gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": achieved_gbs / pk["hbm_gbs"], "traffic": traffic,
                "kernel": kname, "alg_bytes_per_launch": alg_bytes,
                "peak_source": pk["source"] + " (burst copy)"}
    else:
        tf = flops / (attn * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": tf / pk["bf16_tflops"], "traffic": traffic,
                "kernel": kname, "flops_per_launch": flops,
                "peak_source": pk["source"] + " (burst cuBLAS bf16)"}
    qb = wl.q.nbytes
    h2d = qb + wl.k.nbytes + wl.v.nbytes + wl.user_offsets.nbytes + wl.cand_to_user.nbytes
    e2e = P.max_over_ranks(statistics.mean(e2e_ms), dev)
    bc = statistics.mean(bc_ms)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws, "steps": args.steps,
        "repeats": repeats, "timed_steps": n_timed,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": config_block(full, {"parallelism": (
            "one GPU" if ws == 1 else
            f"one batch of {full.n_user} users over {ws} GPUs, whole users with their candidates "
            f"per GPU (longest first, balanced by candidates x keys), no exchange"),
            "global_batch": full.n_cand}),
        "candidates_per_s": P.job_throughput(full.n_cand, ms),
        "pct_of_peak": {"bf16_tensor": value / ws / pk["bf16_tflops"],
                        "hbm_roofline_attn_kernel": achieved_gbs / pk["hbm_gbs"]},
        "kernel_ms": {"plan": statistics.mean(plan_ms), "attn": attn,
                      "step_min": min(step_ms), "step_median": statistics.median(step_ms)},
        "roofline": roof,
        "e2e": {"value": total_flops / (e2e * 1e-3) / 1e12, "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": qb, "ms_per_step": e2e},
        "l2_hot": {"ms_per_step": statistics.mean(hot),
                   "value": flops / (statistics.mean(hot) * 1e-3) / 1e12, "unit": "TFLOP/s",
                   "what": "the same step with no L2 flush between steps (not the headline)"},
        "broadcast_path": {"ms_per_step": bc, "value": flops / (bc * 1e-3) / 1e12, "unit": "TFLOP/s",
                           "ikbo_speedup": bc / ms,
                           "extra_bytes": nums["broadcast_extra_bytes"]},
        "gpu_launches": ikbo.launches_per_call(wl.n_cand, wl.n_user) * n_timed,
        "clocks": clocks,
    }
    if rank == 0:
        line["cpu_baseline"] = cpu_baseline(wl, args.cpu_seconds) if not args.no_cpu_baseline else None
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


def run_fused(args):
    """Fused self + target attention ("In-Kernel Broadcast Optimization", §3.3): the target
    attention of the workload plus the self-attention of every user sequence over itself,
    in one launch; timed beside the same work as two launches (target, then self only)."""
    import torch

    import broadcast_target_attention_gb300 as ikbo

    ws, rank, local = P.dist_env()
    if ws > 1:
        raise SystemExit("--with-self measures one GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ikbo.load()
    ikbo.set_kernel(args.kernel)
    wl = workload_one_gpu(args.config)
    c = wl.cfg
    lens = np.diff(wl.user_offsets.astype(np.int64))
    nums = A.workload_numbers(wl)
    flops = nums["flops"] + A.self_flops(c.H, c.D, lens)
    alg_bytes = nums["alg_bytes"] + A.self_extra_bytes(c.H, c.D, wl.T)
    qu_bits = W.user_queries(wl)

    def t(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a)).view(dt).to(dev)

    q = t(wl.q.view(np.int16), torch.bfloat16)
    qu = t(qu_bits.view(np.int16), torch.bfloat16)
    k = t(wl.k.view(np.int16), torch.bfloat16)
    v = t(wl.v.view(np.int16), torch.bfloat16)
    off = t(wl.user_offsets, torch.int32)
    c2u = t(wl.cand_to_user, torch.int32)
    out, out_user = torch.empty_like(q), torch.empty_like(qu)
    q0, c2u0, out0 = q[:0], c2u[:0], out[:0]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev)

    def fused():
        ikbo.fused_attn_fwd(q, qu, k, v, off, c2u, wl.scale, out=out, out_user=out_user)

    def separate():
        ikbo.attn_fwd(q, k, v, off, c2u, wl.scale, out=out)
        ikbo.fused_attn_fwd(q0, qu, k, v, off, c2u0, wl.scale, out=out0, out_user=out_user)

    def timed(fn, n):
        evs = []
        for i in range(n):
            flush.fill_(i & 0xFF)
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record()
            fn()
            e.record()
            evs.append((s, e))
        torch.cuda.synchronize(dev)
        return [s.elapsed_time(e) for s, e in evs]

    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            flush.fill_(1)
            fused()
            separate()
        assert ikbo.get_device_error() == 0
        torch.cuda.synchronize(dev)
        clk.mark_start()
        fused_ms = timed(fused, args.steps)
        clk.mark_end()
        sep_ms = timed(separate, args.steps)
        # end to end: host tensors copied in, the fused call, both outputs copied back
        hq, hqu, hk, hv = (x.cpu().pin_memory() for x in (q, qu, k, v))
        hoff, hc2u = off.cpu().pin_memory(), c2u.cpu().pin_memory()
        ho, hou = torch.empty_like(hq).pin_memory(), torch.empty_like(hqu).pin_memory()

        def e2e_step():
            dq, dqu, dk, dv = (x.to(dev, non_blocking=True) for x in (hq, hqu, hk, hv))
            doff, dc2u = hoff.to(dev, non_blocking=True), hc2u.to(dev, non_blocking=True)
            o, ou = ikbo.fused_attn_fwd(dq, dqu, dk, dv, doff, dc2u, wl.scale)
            ho.copy_(o, non_blocking=True)
            hou.copy_(ou, non_blocking=True)
            torch.cuda.synchronize(dev)

        for _ in range(3):
            e2e_step()
        e2e_ms = []
        for _ in range(min(args.steps, 50)):
            t0 = time.perf_counter()
            e2e_step()
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
    assert ikbo.get_device_error() == 0
    ms = statistics.mean(fused_ms)
    sep = statistics.mean(sep_ms)
    pk = peaks()
    ai = flops / alg_bytes
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    choice = ikbo.selected_kernel(wl.n_cand, wl.n_user, c.H, c.Lq, c.D, int(wl.user_offsets[-1]))
    kname = f"{ikbo.KERNEL_NAMES[choice]}<{c.D}>"
    if choice == ikbo.KERNEL_TC2:
        kname = kname[:-1] + ", true>"          # the fused instantiation of the two-tile kernel
    traffic = kernel_traffic(kname, c.name)
    if ai < ridge:
        gbs = alg_bytes / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / pk["hbm_gbs"], "traffic": traffic, "kernel": kname,
                "alg_bytes_per_launch": alg_bytes, "peak_source": pk["source"] + " (burst copy)"}
    else:
        tf = flops / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": tf / pk["bf16_tflops"], "traffic": traffic, "kernel": kname,
                "flops_per_launch": flops, "peak_source": pk["source"] + " (burst cuBLAS bf16)"}
    h2d = sum(x.nbytes for x in (wl.q, qu_bits, wl.k, wl.v, wl.user_offsets, wl.cand_to_user))
    d2h = wl.q.nbytes + qu_bits.nbytes
    e2e = statistics.mean(e2e_ms)
    line = {
        "metric": METRIC + " -- fused self + target attention", "value": flops / (ms * 1e-3) / 1e12,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": config_block(wl, {"self_attention": "every user sequence over itself, full, "
                                                      "queries drawn like k (seeded)",
                                    "self_flops": A.self_flops(c.H, c.D, lens),
                                    "target_flops": nums["flops"]}),
        "roofline": roof,
        "fusion": {"fused_ms": ms, "separate_ms": sep, "speedup": sep / ms,
                   "separate": "target call, then a self-only call of the same kernel"},
        "e2e": {"value": flops / (e2e * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e},
        "gpu_launches": args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


def run_lce(args):
    """IKBO linear compression ("In-Kernel Broadcast Optimization", §2) on one GPU, timed
    beside the broadcast form it replaces (the user block copied to every candidate, then one
    batched product through torch / cuBLAS)."""
    import torch

    import broadcast_target_attention_gb300 as ikbo

    ws, rank, local = P.dist_env()
    if ws > 1:
        raise SystemExit("--lce measures one GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ikbo.load()
    wl = W.lce_generate(W.LCE_CONFIGS[args.lce])
    c = wl.cfg
    ku, kc = wl.X_user.shape[1], wl.X_cand.shape[1]
    flops = A.lce_flops(c.M, c.N, c.n_user, c.K_user, c.n_cand, c.K_cand)
    alg_bytes = A.lce_alg_bytes(c.M, c.N, c.n_user, ku, c.n_cand, kc)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    Wu, Wc, Xu, Xc = bf(wl.W_user), bf(wl.W_cand), bf(wl.X_user), bf(wl.X_cand)
    c2u = torch.from_numpy(wl.cand_to_user).to(dev)
    out = torch.empty((c.n_cand, c.M, c.N), dtype=torch.bfloat16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev)
    Wfull = torch.cat([Wu, Wc], dim=1)

    def ikbo_step():
        ikbo.lce_fwd(Wu, Wc, Xu, Xc, c2u, out=out)

    def broadcast_step():
        X = torch.cat([Xu[c2u.long()], Xc], dim=1)          # the materialised broadcast
        return torch.matmul(Wfull, X)

    def timed(fn, n):
        evs = []
        for i in range(n):
            flush.fill_(i & 0xFF)
            s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s_.record()
            fn()
            e_.record()
            evs.append((s_, e_))
        torch.cuda.synchronize(dev)
        return [a.elapsed_time(b) for a, b in evs]

    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            flush.fill_(1)
            ikbo_step()
            broadcast_step()
        assert ikbo.get_device_error() == 0
        torch.cuda.synchronize(dev)
        clk.mark_start()
        ms_list = timed(ikbo_step, args.steps)
        clk.mark_end()
        bc_list = timed(broadcast_step, min(args.steps, 20))
        # per-kernel times: the user stage and the candidate stage (events around each launch)
        ikbo.set_timing(True)
        st0, st1 = [], []
        for i in range(min(args.steps, 50)):
            flush.fill_(i & 0xFF)
            ikbo_step()
            a_, b_ = ikbo.get_timing()
            st0.append(a_)
            st1.append(b_)
        ikbo.set_timing(False)
        # end to end: host tensors copied in, the call, the output copied back
        hWu, hWc, hXu, hXc, hc2u = (x.cpu().pin_memory() for x in (Wu, Wc, Xu, Xc, c2u))
        hout = torch.empty_like(out, device="cpu").pin_memory()

        def e2e_step():
            d = [x.to(dev, non_blocking=True) for x in (hWu, hWc, hXu, hXc, hc2u)]
            o = ikbo.lce_fwd(*d)
            hout.copy_(o, non_blocking=True)
            torch.cuda.synchronize(dev)

        for _ in range(3):
            e2e_step()
        e2e_ms = []
        for _ in range(min(args.steps, 20)):
            t0 = time.perf_counter()
            e2e_step()
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
    assert ikbo.get_device_error() == 0
    ms = statistics.mean(ms_list)
    bc = statistics.mean(bc_list)
    pk = peaks()
    tf = flops / (ms * 1e-3) / 1e12
    ai = flops / alg_bytes
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    gbs = alg_bytes / (ms * 1e-3) / 1e9
    kname = lce_kernel_name(c.M, c.N)
    # DRAM bytes of the candidate stage (the launch that moves all but ~2 % of the bytes)
    traffic = kernel_traffic(kname, c.name)
    if ai < ridge:
        roof = {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / pk["hbm_gbs"], "traffic": traffic, "kernel": kname,
                "alg_bytes_per_launch": alg_bytes, "peak_source": pk["source"] + " (burst copy)"}
    else:
        roof = {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                "frac": tf / pk["bf16_tflops"], "traffic": traffic, "kernel": kname,
                "flops_per_launch": flops, "peak_source": pk["source"] + " (burst cuBLAS bf16)"}
    h2d = sum(x.nbytes for x in (wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user))
    e2e = statistics.mean(e2e_ms)
    line = {
        "metric": "IKBO linear compression BF16 TFLOP/s (decomposed work)", "value": tf,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{c.name}: {c.description}", "n_cand": c.n_cand, "n_user": c.n_user,
                   "M": c.M, "K_user": c.K_user, "K_cand": c.K_cand, "N": c.N,
                   "l2": "flushed before every timed step (write of 2x L2 size)",
                   "ai_flop_per_byte": ai},
        "kernel_ms": {"user_stage": statistics.mean(st0), "candidate_stage": statistics.mean(st1)},
        "roofline": roof,
        "broadcast_path": {"ms_per_step": bc, "ikbo_speedup": bc / ms,
                           "what": "torch: X = cat(X_user[cand_to_user], X_cand); matmul(W, X)"},
        "e2e": {"value": flops / (e2e * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": int(out.numel() * 2), "ms_per_step": e2e},
        "gpu_launches": 2 * args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


def _timed(fn, n, flush, dev):
    """CUDA-event times (ms) of n calls of fn, L2 flushed before each."""
    import torch
    evs = []
    for i in range(n):
        flush.fill_(i & 0xFF)
        s_, e_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_.record()
        fn()
        e_.record()
        evs.append((s_, e_))
    torch.cuda.synchronize(dev)
    return [a.elapsed_time(b) for a, b in evs]


def _roofline(flops, alg_bytes, ms, kname, traffic=None):
    pk = peaks()
    ai = flops / alg_bytes
    ridge = pk["bf16_tflops"] * 1e12 / (pk["hbm_gbs"] * 1e9)
    if ai < ridge:
        gbs = alg_bytes / (ms * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"], "unit": "GB/s",
                "frac": gbs / pk["hbm_gbs"], "traffic": traffic, "kernel": kname,
                "alg_bytes_per_launch": alg_bytes, "peak_source": pk["source"] + " (burst copy)"}
    tf = flops / (ms * 1e-3) / 1e12
    return {"bound": "tensor", "achieved": tf, "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
            "frac": tf / pk["bf16_tflops"], "traffic": traffic, "kernel": kname,
            "flops_per_launch": flops, "peak_source": pk["source"] + " (burst cuBLAS bf16)"}


def run_ml(args):
    """Target attention over a user -> vendor -> item hierarchy ("In-Kernel Broadcast
    Optimization", §5): the library walks item_to_vendor and vendor_to_user itself; timed
    beside the two-level call given the per-item user map."""
    import torch

    import broadcast_target_attention_gb300 as ikbo

    ws, rank, local = P.dist_env()
    if ws > 1:
        raise SystemExit("--ml measures one GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ikbo.load()
    m = W.ml_generate(W.ML_CONFIGS[args.ml])
    wl, c = m.wl, m.cfg
    nums = A.workload_numbers(wl)
    flops = nums["flops"]
    alg_bytes = nums["alg_bytes"] + 4 * c.n_vendor     # the vendor map as well

    def t(a, dt):
        return torch.from_numpy(np.ascontiguousarray(a)).view(dt).to(dev)

    q, k, v = (t(x.view(np.int16), torch.bfloat16) for x in (wl.q, wl.k, wl.v))
    off = t(wl.user_offsets, torch.int32)
    i2v, v2u = t(m.item_to_vendor, torch.int32), t(m.vendor_to_user, torch.int32)
    item_user = t(wl.cand_to_user, torch.int32)
    out = torch.empty_like(q)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev)

    def ml_step():
        ikbo.ml_attn_fwd(q, k, v, off, i2v, v2u, wl.scale, out=out)

    def two_level_step():
        ikbo.attn_fwd(q, k, v, off, item_user, wl.scale, out=out)

    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            flush.fill_(1)
            ml_step()
            two_level_step()
        assert ikbo.get_device_error() == 0
        torch.cuda.synchronize(dev)
        clk.mark_start()
        ms_list = _timed(ml_step, args.steps, flush, dev)
        clk.mark_end()
        two_ms = _timed(two_level_step, args.steps, flush, dev)
        ikbo.set_timing(True)
        kern = []
        for i in range(min(args.steps, 50)):
            flush.fill_(i & 0xFF)
            ml_step()
            kern.append(ikbo.get_timing()[1])
        ikbo.set_timing(False)
        hq, hk, hv = (x.cpu().pin_memory() for x in (q, k, v))
        hoff, hi2v, hv2u = (x.cpu().pin_memory() for x in (off, i2v, v2u))
        hout = torch.empty_like(hq).pin_memory()

        def e2e_step():
            d = [x.to(dev, non_blocking=True) for x in (hq, hk, hv, hoff, hi2v, hv2u)]
            o = ikbo.ml_attn_fwd(*d, wl.scale)
            hout.copy_(o, non_blocking=True)
            torch.cuda.synchronize(dev)

        for _ in range(3):
            e2e_step()
        e2e_ms = []
        for _ in range(min(args.steps, 50)):
            t0 = time.perf_counter()
            e2e_step()
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
    assert ikbo.get_device_error() == 0
    ms = statistics.mean(ms_list)
    kms = statistics.mean(kern)
    kname = f"{ikbo.KERNEL_NAMES[ikbo.selected_kernel(wl.n_cand, wl.n_user, c.H, c.Lq, c.D)]}<{c.D}>"
    h2d = sum(x.nbytes for x in (wl.q, wl.k, wl.v, wl.user_offsets, m.item_to_vendor, m.vendor_to_user))
    e2e = statistics.mean(e2e_ms)
    line = {
        "metric": METRIC + " -- user -> vendor -> item hierarchy", "value": flops / (ms * 1e-3) / 1e12,
        "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": config_block(wl, {"workload": f"{c.name}: {c.description}", "n_item": c.n_item,
                                    "n_vendor": c.n_vendor}),
        "kernel_ms": {"attn": kms},
        "roofline": _roofline(flops, alg_bytes, kms, kname),
        "two_level_call": {"ms_per_step": statistics.mean(two_ms),
                           "what": "ikbo_attn_fwd given the per-item user map (walked by the caller)"},
        "e2e": {"value": flops / (e2e * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": wl.q.nbytes, "ms_per_step": e2e},
        "gpu_launches": ikbo.launches_per_call(wl.n_cand, wl.n_user) * args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


def run_ml_lce(args):
    """Linear compression over a user -> vendor -> item hierarchy: one launch per level, each
    level's product once per entry of that level; timed beside the broadcast form (both
    blocks copied to every item, then one batched product through torch / cuBLAS)."""
    import torch

    import broadcast_target_attention_gb300 as ikbo

    ws, rank, local = P.dist_env()
    if ws > 1:
        raise SystemExit("--lce-ml measures one GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ikbo.load()
    l = W.lce_ml_generate(W.LCE_ML_CONFIGS[args.lce_ml])
    c = l.cfg
    ku, kv, ki = l.X_user.shape[1], l.X_vendor.shape[1], l.X_item.shape[1]
    flops = A.ml_lce_flops(c.M, c.N, c.n_user, c.K_user, c.n_vendor, c.K_vendor, c.n_item, c.K_item)
    alg_bytes = A.ml_lce_alg_bytes(c.M, c.N, c.n_user, ku, c.n_vendor, kv, c.n_item, ki)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(dev)
    Wu, Wv, Wi, Xu, Xv, Xi = (bf(x) for x in (l.W_user, l.W_vendor, l.W_item, l.X_user, l.X_vendor,
                                              l.X_item))
    i2v, v2u = (torch.from_numpy(x).to(dev) for x in (l.item_to_vendor, l.vendor_to_user))
    item_user = torch.from_numpy(l.item_user).to(dev).long()
    out = torch.empty((c.n_item, c.M, c.N), dtype=torch.bfloat16, device=dev)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev)
    Wfull = torch.cat([Wu, Wv, Wi], dim=1)

    def ikbo_step():
        ikbo.ml_lce_fwd(Wu, Wv, Wi, Xu, Xv, Xi, i2v, v2u, out=out)

    def broadcast_step():
        X = torch.cat([Xu[item_user], Xv[i2v.long()], Xi], dim=1)   # the materialised broadcast
        return torch.matmul(Wfull, X)

    with ClockSampler(local) as clk:
        for _ in range(args.warmup):
            flush.fill_(1)
            ikbo_step()
            broadcast_step()
        assert ikbo.get_device_error() == 0
        torch.cuda.synchronize(dev)
        clk.mark_start()
        ms_list = _timed(ikbo_step, args.steps, flush, dev)
        clk.mark_end()
        bc_list = _timed(broadcast_step, min(args.steps, 20), flush, dev)
        host = [x.cpu().pin_memory() for x in (Wu, Wv, Wi, Xu, Xv, Xi, i2v, v2u)]
        hout = torch.empty_like(out, device="cpu").pin_memory()

        def e2e_step():
            d = [x.to(dev, non_blocking=True) for x in host]
            o = ikbo.ml_lce_fwd(*d)
            hout.copy_(o, non_blocking=True)
            torch.cuda.synchronize(dev)

        for _ in range(3):
            e2e_step()
        e2e_ms = []
        for _ in range(min(args.steps, 20)):
            t0 = time.perf_counter()
            e2e_step()
            e2e_ms.append((time.perf_counter() - t0) * 1e3)
    assert ikbo.get_device_error() == 0
    ms = statistics.mean(ms_list)
    bc = statistics.mean(bc_list)
    tf = flops / (ms * 1e-3) / 1e12
    h2d = sum(x.nbytes for x in (l.W_user, l.W_vendor, l.W_item, l.X_user, l.X_vendor, l.X_item,
                                 l.item_to_vendor, l.vendor_to_user))
    e2e = statistics.mean(e2e_ms)
    line = {
        "metric": "IKBO linear compression BF16 TFLOP/s (decomposed work) -- user -> vendor -> item",
        "value": tf, "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{c.name}: {c.description}", "n_item": c.n_item,
                   "n_vendor": c.n_vendor, "n_user": c.n_user, "M": c.M, "K_user": c.K_user,
                   "K_vendor": c.K_vendor, "K_item": c.K_item, "N": c.N,
                   "l2": "flushed before every timed step (write of 2x L2 size)",
                   "ai_flop_per_byte": flops / alg_bytes},
        "roofline": _roofline(flops, alg_bytes, ms, lce_kernel_name(c.M, c.N)),
        "broadcast_path": {"ms_per_step": bc, "ikbo_speedup": bc / ms,
                           "what": "torch: X = cat(X_user[u], X_vendor[v], X_item); matmul(W, X)"},
        "e2e": {"value": flops / (e2e * 1e-3) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": int(out.numel() * 2), "ms_per_step": e2e},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
        "cpu_baseline": None,
    }
    print(json.dumps(line), flush=True)


# Candidate-to-user ratios of the sweep ("In-Kernel Broadcast Optimization", §4: IKBO was
# validated from about 10,000:1 down to 10:1; the benefit grows with the ratio).
RATIO_SWEEP = ((4096, 4096), (4096, 410), (4096, 41), (4096, 4), (10000, 1))


def run_ratio_sweep(args):
    """IKBO against the explicit-broadcast path over candidate-to-user ratios at one shape
    (H=4, D=128, Lq=1, L ~ U[256, 1024]): one JSON line per ratio, each step timed between
    events with the L2 flushed before it."""
    import torch

    import broadcast_target_attention_gb300 as ikbo

    ws, rank, local = P.dist_env()
    if ws > 1:
        raise SystemExit("--ratio-sweep measures one GPU")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ikbo.load()
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2 // 4 + 1024, dtype=torch.int32, device=dev)
    for n_cand, n_user in RATIO_SWEEP:
        cfg = W.Config(name=f"ratio_{n_cand}x{n_user}", n_cand=n_cand, n_user=n_user, H=4, D=128,
                       Lq=1, seed=7, counts="multinomial", lens="uniform", len_lo=256, len_hi=1024,
                       description=f"{n_cand} candidates over {n_user} users, L~U[256,1024], "
                                   "H=4 D=128 Lq=1")
        wl = W.generate(cfg)
        nums = A.workload_numbers(wl)
        t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).view(dt).to(dev)
        q, k, v = (t(x.view(np.int16), torch.bfloat16) for x in (wl.q, wl.k, wl.v))
        off, c2u = t(wl.user_offsets, torch.int32), t(wl.cand_to_user, torch.int32)
        out = torch.empty_like(q)
        ikbo_step = lambda: ikbo.attn_fwd(q, k, v, off, c2u, wl.scale, out=out)
        bc_step = lambda: ikbo.broadcast_attn_fwd(q, k, v, off, c2u, wl.scale, out=out)
        for _ in range(args.warmup):
            flush.fill_(1)
            ikbo_step()
            bc_step()
        assert ikbo.get_device_error() == 0
        ms = statistics.mean(_timed(ikbo_step, args.steps, flush, dev))
        bc = statistics.mean(_timed(bc_step, min(args.steps, 10), flush, dev))
        kname = f"{ikbo.KERNEL_NAMES[ikbo.selected_kernel(n_cand, n_user, 4, 1, 128)]}<128>"
        line = {
            "metric": METRIC + " -- candidate-to-user ratio sweep",
            "value": nums["flops"] / (ms * 1e-3) / 1e12, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_block(wl, {"ratio": n_cand / n_user}),
            "roofline": _roofline(nums["flops"], nums["alg_bytes"], ms, kname),
            "broadcast_path": {"ms_per_step": bc, "ikbo_speedup": bc / ms,
                               "extra_bytes": nums["broadcast_extra_bytes"]},
            "gpu_launches": ikbo.launches_per_call(n_cand, n_user) * args.steps,
        }
        print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="ikbo", choices=["ikbo", "reference"])
    ap.add_argument("--config", default=W.HEADLINE, choices=sorted(W.CONFIGS) + sorted(W.LONG_CONFIGS))
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--kernel", type=int, default=0, choices=[0, 1, 2, 3, 4],
                    help="attention kernel (ikbo_set_kernel): 0 = the automatic choice")
    ap.add_argument("--min-timed-s", type=float, default=0.25,
                    help="repeat the block of --steps timed steps until it lasts this long")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--lce", default=None, choices=sorted(W.LCE_CONFIGS),
                    help="measure IKBO linear compression on this workload instead")
    ap.add_argument("--with-self", action="store_true",
                    help="measure the fused self + target attention of the workload instead")
    ap.add_argument("--ml", default=None, choices=sorted(W.ML_CONFIGS),
                    help="measure target attention over a user -> vendor -> item hierarchy")
    ap.add_argument("--lce-ml", default=None, choices=sorted(W.LCE_ML_CONFIGS),
                    help="measure linear compression over a user -> vendor -> item hierarchy")
    ap.add_argument("--ratio-sweep", action="store_true",
                    help="IKBO against the broadcast path over candidate-to-user ratios")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.lce:
        run_lce(args)
    elif args.with_self:
        run_fused(args)
    elif args.ml:
        run_ml(args)
    elif args.lce_ml:
        run_ml_lce(args)
    elif args.ratio_sweep:
        run_ratio_sweep(args)
    else:
        run_ikbo(args)


if __name__ == "__main__":
    main()
