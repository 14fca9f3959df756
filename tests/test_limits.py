"""Parity at the size limits of the planning: exactly the largest batch the attention kernels
plan in-kernel (20480 candidates, 1024 users: the shared-memory scratch full), sorted and
unsorted, and one past each limit (the planning kernel's work list, read by the one-tile
kernel; the two-tile choice falls back to it).  Sampled candidates against the oracle."""
import numpy as np
import pytest

import oracle
from broadcast_target_attention_gb300 import workloads as W
from _helpers import assert_close, out_f64, to_device

pytestmark = pytest.mark.gpu


def limit_workload(n_cand, n_user, shuffle, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    counts = 1 + rng.multinomial(n_cand - n_user, np.full(n_user, 1.0 / n_user))
    lens = rng.integers(0, 97, size=n_user)           # empty sequences included
    return W.custom(n_user=n_user, counts=counts.tolist(), lens=lens.tolist(), H=1, D=64, Lq=1,
                    seed=seed, shuffle=shuffle)


@pytest.mark.parametrize("n_cand,n_user,launches", [(20480, 1024, 1), (20481, 1024, 2),
                                                     (20480, 1025, 2)])
@pytest.mark.parametrize("shuffle", [False, True])
@pytest.mark.parametrize("kernel", [0, 3, 4])
def test_planning_limits(gpu_lib, n_cand, n_user, launches, shuffle, kernel):
    wl = limit_workload(n_cand, n_user, shuffle, seed=n_cand + n_user)
    assert gpu_lib.launches_per_call(n_cand, n_user) == launches
    d = to_device(wl)
    prev = gpu_lib.set_kernel(kernel)
    try:
        out = gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale)
        rc = gpu_lib.get_device_error()
    finally:
        gpu_lib.set_kernel(prev)
    assert rc == 0
    cands = W.sample_candidates(wl, 200)
    what = f"{n_cand}x{n_user} shuffle={shuffle} kernel={kernel}"
    assert_close(out_f64(out, cands), oracle.attention_wl(wl, cands), what)
    # the rows of candidates whose user has no keys are zero
    empty = np.nonzero(np.diff(wl.user_offsets) == 0)[0]
    hit = np.nonzero(np.isin(wl.cand_to_user, empty))[0][:50]
    if hit.size:
        assert np.all(out_f64(out, hit) == 0), what
