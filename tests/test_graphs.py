"""The library's calls inside CUDA graphs: a call captured on a stream (its stream-ordered
scratch allocation, and for the planning-kernel and linear-compression paths the programmatic
dependent launch, become graph nodes) and replayed, against the fp64 oracle; replays follow
new contents of the same input buffers.  The first call of each kind runs outside the
capture (it sets the device's kernel attributes up)."""
import numpy as np
import pytest
import torch

import oracle
from broadcast_target_attention_gb300 import workloads as W
from _helpers import assert_close, out_f64, to_device

pytestmark = pytest.mark.gpu


def capture(fn):
    fn()                                    # set-up outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    return g


@pytest.mark.parametrize("entry", ["attn_fwd", "attn_fwd_noalloc"])
@pytest.mark.parametrize("n_cand,n_user", [(300, 7), (20481, 64)])   # in-kernel planning; planning kernel
def test_attention_graph_replay(gpu_lib, entry, n_cand, n_user):
    rng = np.random.Generator(np.random.PCG64(n_cand))
    counts = 1 + rng.multinomial(n_cand - n_user, np.full(n_user, 1.0 / n_user))
    lens = rng.integers(1, 300, size=n_user)
    wl = W.custom(n_user=n_user, counts=counts.tolist(), lens=lens.tolist(), H=2, D=64, Lq=1,
                  seed=n_user)
    d = to_device(wl)
    out = torch.empty_like(d["q"])
    call = getattr(gpu_lib, entry)
    g = capture(lambda: call(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale,
                             out=out))
    cands = W.sample_candidates(wl, 128)
    for rep in range(2):
        if rep == 1:
            # new queries in the captured buffer: the replay reads them
            wl.q = W.custom(n_user=n_user, counts=counts.tolist(), lens=lens.tolist(), H=2, D=64,
                            Lq=1, seed=n_user + 1).q
            d["q"].copy_(to_device(wl)["q"])
        out.fill_(7.0)
        g.replay()
        torch.cuda.synchronize()
        assert gpu_lib.get_device_error() == 0
        assert_close(out_f64(out, cands), oracle.attention_wl(wl, cands), f"{entry} replay {rep}")


def test_two_tile_kernel_graph_replay(gpu_lib):
    wl = W.custom(n_user=2, counts=[600, 300], lens=[700, 260], H=4, D=128, Lq=2, seed=8)
    d = to_device(wl)
    out = torch.empty_like(d["q"])
    prev = gpu_lib.set_kernel(gpu_lib.KERNEL_TC2)
    try:
        g = capture(lambda: gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"],
                                             d["cand_to_user"], wl.scale, out=out))
    finally:
        gpu_lib.set_kernel(prev)
    g.replay()
    torch.cuda.synchronize()
    assert gpu_lib.get_device_error() == 0
    cands = W.sample_candidates(wl, 96)
    assert_close(out_f64(out, cands), oracle.attention_wl(wl, cands), "two-tile replay")


def test_linear_compression_graph_replay(gpu_lib):
    """Two launches, the second a programmatic dependent of the first."""
    cfg = W.LceConfig(name="g", n_cand=13, n_user=4, M=200, K_user=64, K_cand=72, N=128, seed=9)
    wl = W.lce_generate(cfg)
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    Wu, Wc, Xu, Xc = bf(wl.W_user), bf(wl.W_cand), bf(wl.X_user), bf(wl.X_cand)
    c2u = torch.from_numpy(wl.cand_to_user).cuda()
    out = torch.empty((cfg.n_cand, cfg.M, cfg.N), dtype=torch.bfloat16, device="cuda")
    g = capture(lambda: gpu_lib.lce_fwd(Wu, Wc, Xu, Xc, c2u, out=out))
    out.fill_(3.0)
    g.replay()
    torch.cuda.synchronize()
    assert gpu_lib.get_device_error() == 0
    ref = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, "lce replay")
