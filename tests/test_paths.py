"""The other entry points on the GPU: the explicit-broadcast comparison path,
the host-buffer path, device-side error reporting, bounded waits, timing."""
import numpy as np
import pytest
import torch

import oracle
from broadcast_target_attention_gb300 import _lib
from broadcast_target_attention_gb300 import workloads as W
from _helpers import assert_close, out_f64, to_device

pytestmark = pytest.mark.gpu


def test_broadcast_path_matches_oracle_in_several_chunks(gpu_lib):
    wl = W.custom(n_user=4, counts=[9, 4, 1, 6], lens=[300, 129, 17, 640], H=2, D=128, Lq=2, seed=4)
    d = to_device(wl)
    row_bytes = 2 * 128 * 2
    budget = 2 * 700 * row_bytes * 2        # about two candidates' copies per chunk
    out = gpu_lib.broadcast_attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"],
                                     wl.scale, mem_budget_bytes=budget)
    assert gpu_lib.get_device_error() == 0
    assert_close(out_f64(out), oracle.attention_wl(wl), "broadcast path")


def test_broadcast_path_rejects_a_budget_below_one_copy(gpu_lib):
    wl = W.custom(n_user=1, counts=[2], lens=[100], H=1, D=64, Lq=1)
    d = to_device(wl)
    with pytest.raises(gpu_lib.IkboError) as e:
        gpu_lib.broadcast_attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"],
                                   wl.scale, mem_budget_bytes=1000)
    assert e.value.status == _lib.IKBO_ERR_BUDGET


def _host_call(gpu_lib, wl):
    d = to_device(wl)
    h = {k_: v_.cpu().pin_memory() for k_, v_ in d.items()}
    host_out = torch.full_like(h["q"], 7.0).pin_memory()
    gpu_lib.attn_fwd_host(h["q"], h["k"], h["v"], h["user_offsets"], h["cand_to_user"], wl.scale,
                          out=host_out)
    return d, host_out


def test_host_path_equals_device_path(gpu_lib):
    """The host path copies in, runs the device path's kernels and copies out: bit-equal."""
    wl = W.generate(W.CONFIGS["ratio_1024x15"])
    d, host_out = _host_call(gpu_lib, wl)
    dev_out = gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale)
    assert torch.equal(host_out, dev_out.cpu())


HOST_CASES = {
    # an empty sequence and users without candidates
    "gaps": dict(n_user=5, counts=[30, 9, 0, 0, 41], lens=[2500, 0, 2600, 100, 2400]),
    # one user with most of the keys
    "first_heavy": dict(n_user=4, counts=[7, 100, 3, 1], lens=[9000, 300, 129, 1]),
}


@pytest.mark.parametrize("case", sorted(HOST_CASES))
@pytest.mark.parametrize("shuffle", [False, True])
def test_host_path_matches_oracle(gpu_lib, case, shuffle):
    wl = W.custom(H=4, D=128, Lq=1, seed=len(case), shuffle=shuffle, **HOST_CASES[case])
    _, host_out = _host_call(gpu_lib, wl)
    cands = W.sample_candidates(wl, 200)
    assert_close(host_out.float().numpy().astype(np.float64)[cands], oracle.attention_wl(wl, cands),
                 f"host path {case} shuffle={shuffle}")


def _sentinel_call(gpu_lib, wl, c2u=None, off=None):
    d = to_device(wl)
    if c2u is not None:
        d["cand_to_user"] = torch.tensor(c2u, dtype=torch.int32, device="cuda")
    if off is not None:
        d["user_offsets"] = torch.tensor(off, dtype=torch.int32, device="cuda")
    out = torch.full_like(d["q"], 7.0)
    gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale, out=out)
    return gpu_lib.get_device_error(), out


@pytest.mark.parametrize("kernel", [1, 2, 3])
def test_bad_candidate_index_is_reported_not_trapped(gpu_lib, kernel):
    wl = W.custom(n_user=2, counts=[2, 2], lens=[10, 20], H=2, D=64, Lq=1)
    prev = gpu_lib.set_kernel(kernel)
    try:
        rc, out = _sentinel_call(gpu_lib, wl, c2u=[0, 1, 2, 1])
    finally:
        gpu_lib.set_kernel(prev)
    assert rc == _lib.IKBO_ERR_INDEX
    assert bool((out == 7.0).all())          # nothing written
    assert gpu_lib.get_device_error() == 0   # the word was cleared


def test_errors_are_kept_per_stream(gpu_lib):
    """An index error of a call on one stream is reported on that stream only: a caller on
    another stream sees its own clean calls, before and after, and the word is cleared."""
    wl = W.custom(n_user=2, counts=[2, 2], lens=[10, 20], H=2, D=64, Lq=1)
    d = to_device(wl)
    bad = torch.tensor([0, 1, 2, 1], dtype=torch.int32, device="cuda")
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    out_a = torch.full_like(d["q"], 7.0)
    with torch.cuda.stream(sa):
        gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], bad, wl.scale, out=out_a)
    with torch.cuda.stream(sb):
        out_b = gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale)
    assert gpu_lib.get_device_error(sb) == 0
    assert gpu_lib.get_device_error(sa) == _lib.IKBO_ERR_INDEX
    assert gpu_lib.get_device_error(sa) == 0
    assert bool((out_a == 7.0).all())
    assert_close(out_f64(out_b), oracle.attention_wl(wl), "clean call on the other stream")
    # the legacy default stream keeps its own word too
    assert gpu_lib.get_device_error(torch.cuda.default_stream()) == 0


def test_bad_offsets_are_reported(gpu_lib):
    wl = W.custom(n_user=2, counts=[2, 2], lens=[10, 20], H=2, D=64, Lq=1)
    rc, out = _sentinel_call(gpu_lib, wl, off=[0, 25, 20])
    assert rc == _lib.IKBO_ERR_OFFSETS
    assert bool((out == 7.0).all())
    rc, _ = _sentinel_call(gpu_lib, wl, off=[3, 13, 33])
    assert rc == _lib.IKBO_ERR_OFFSETS


@pytest.mark.parametrize("kernel", [2, 3])
def test_bounded_wait_reports_timeout_and_context_survives(gpu_lib, kernel):
    """The producer is told never to arm the query barrier: every waiting warp
    gives up after 50 ms, the kernel exits normally and reports the timeout."""
    wl = W.custom(n_user=2, counts=[5, 3], lens=[300, 40], H=2, D=128, Lq=1, seed=5)
    gpu_lib.set_debug(1, 50_000_000)
    prev = gpu_lib.set_kernel(kernel)
    try:
        rc, _ = _sentinel_call(gpu_lib, wl)
    finally:
        gpu_lib.set_debug(0, 0)
        gpu_lib.set_kernel(prev)
    assert rc == _lib.IKBO_ERR_TIMEOUT
    rc, out = _sentinel_call(gpu_lib, wl)     # the context is still usable
    assert rc == 0
    assert_close(out_f64(out), oracle.attention_wl(wl), "after timeout")


def test_timing_hooks(gpu_lib):
    wl = W.generate(W.CONFIGS["ratio_1024x15"])
    d = to_device(wl)
    gpu_lib.set_timing(True)
    try:
        gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale)
        plan_ms, attn_ms = gpu_lib.get_timing()
    finally:
        gpu_lib.set_timing(False)
    assert plan_ms > 0 and attn_ms > 0


def test_shutdown_then_calls_again(gpu_lib):
    """ikbo_shutdown releases the per-device state and trims the pool; the next calls set the
    device up again and give the same results."""
    wl = W.custom(n_user=3, counts=[40, 3, 70], lens=[300, 129, 500], H=2, D=128, Lq=1, seed=12)
    d = to_device(wl)
    first = gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale)
    gpu_lib.set_timing(True)
    gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale)
    gpu_lib.set_timing(False)
    assert gpu_lib.get_device_error() == 0
    gpu_lib.shutdown()
    gpu_lib.shutdown()                                   # again: nothing left to release
    again = gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale)
    assert gpu_lib.get_device_error() == 0
    assert torch.equal(first, again)
    h = {k_: v_.cpu().pin_memory() for k_, v_ in d.items()}
    host_out = torch.empty_like(h["q"]).pin_memory()
    gpu_lib.attn_fwd_host(h["q"], h["k"], h["v"], h["user_offsets"], h["cand_to_user"], wl.scale,
                          out=host_out)
    assert torch.equal(host_out, first.cpu())
