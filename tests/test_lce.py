"""IKBO linear compression ("In-Kernel Broadcast Optimization", §2) through the C ABI.

CPU: host-side argument checks (nothing reaches the GPU).  GPU: the tcgen05 path against
the fp64 oracle on the pages' configuration (sampled candidates) and on small cases that
cover ragged M (a partial last row tile), K blocks that are not multiples of 64, every
supported N (N = 128 and 256 with M over one row tile run on CTA pairs with M = 256
MMAs, the others CTA by CTA), a call without a user block, one candidate per user, and
a bad index.
"""
import numpy as np
import pytest
import torch

import oracle
from broadcast_target_attention_gb300 import _lib
from broadcast_target_attention_gb300 import build as B
from broadcast_target_attention_gb300 import workloads as W
from _helpers import assert_close


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.lib()


def test_host_checks(lib):
    f = lib.ikbo_lce_fwd
    big = 1 << 40   # a fake, aligned address: every case below is refused before it is used
    assert f(big, big, big, big, big, 4, 2, 16, 12, 16, 64, big, None) == _lib.IKBO_ERR_SHAPE  # K_user % 8
    assert f(big, big, big, big, big, 4, 2, 16, 16, 0, 64, big, None) == _lib.IKBO_ERR_SHAPE   # K_cand < 8
    assert f(big, big, big, big, big, 4, 2, 16, 16, 16, 96, big, None) == _lib.IKBO_ERR_SHAPE  # N % 64
    assert f(big, big, big, big, big, 4, 2, 16, 16, 16, 320, big, None) == _lib.IKBO_ERR_SHAPE
    assert f(big, big, big, big, big, 4, 2, 0, 16, 16, 64, big, None) == _lib.IKBO_ERR_SHAPE   # M < 1
    assert f(big, big, big, big, big, -1, 2, 16, 16, 16, 64, big, None) == _lib.IKBO_ERR_SHAPE
    assert f(big, big, big, big, big, 0, 2, 16, 16, 16, 64, big, None) == 0                     # empty batch
    assert f(big, None, big, big, big, 4, 2, 16, 16, 16, 64, big, None) == _lib.IKBO_ERR_NULL
    assert f(None, big, None, big, None, 4, 2, 16, 16, 16, 64, big, None) == _lib.IKBO_ERR_NULL  # user block, no W_user
    assert f(big, big + 8, big, big, big, 4, 2, 16, 16, 16, 64, big + 4096, None) == _lib.IKBO_ERR_ALIGN
    assert f(big, big, big, big, big, 4, 0, 16, 16, 16, 64, big + 4096, None) == _lib.IKBO_ERR_INDEX
    # out overlapping X_cand
    assert f(big, big, big, big + (1 << 20), big, 4, 2, 16, 16, 16, 64, big + (1 << 20), None) == \
        _lib.IKBO_ERR_ALIAS


def to_dev(wl):
    t = lambda a, dt: torch.from_numpy(np.ascontiguousarray(a)).view(dt).cuda()
    bf = lambda a: t(a.view(np.int16), torch.bfloat16)
    return bf(wl.W_user), bf(wl.W_cand), bf(wl.X_user), bf(wl.X_cand), t(wl.cand_to_user, torch.int32)


def run(ikbo, wl):
    Wu, Wc, Xu, Xc, c2u = to_dev(wl)
    out = ikbo.lce_fwd(Wu, Wc, Xu, Xc, c2u)
    assert ikbo.get_device_error() == 0
    return out


def check(ikbo, wl, what, cands=None):
    out = run(ikbo, wl)
    got = out.float().cpu().numpy().astype(np.float64)
    if cands is not None:
        got = got[cands]
    ref = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user, cands)
    assert_close(got, ref, what)


@pytest.mark.gpu
def test_pages_configuration(gpu_lib):
    wl = W.lce_generate(W.LCE_CONFIGS["lce_1024x15"])
    c2u = wl.cand_to_user
    cands = np.unique(np.concatenate([np.linspace(0, wl.cfg.n_cand - 1, 40).astype(np.int64),
                                      np.searchsorted(c2u, np.arange(wl.cfg.n_user))]))
    check(gpu_lib, wl, "lce_1024x15", cands)


@pytest.mark.gpu
def test_tiny(gpu_lib):
    check(gpu_lib, W.lce_generate(W.LCE_CONFIGS["lce_tiny_8x3"]), "lce_tiny_8x3")


@pytest.mark.gpu
@pytest.mark.parametrize("N", [64, 128, 192, 256])
@pytest.mark.parametrize("M,K_user,K_cand", [(1, 8, 8), (130, 72, 136), (257, 200, 64)])
def test_shapes(gpu_lib, M, K_user, K_cand, N):
    cfg = W.LceConfig(name="s", n_cand=11, n_user=4, M=M, K_user=K_user, K_cand=K_cand, N=N, seed=M + N)
    check(gpu_lib, W.lce_generate(cfg), f"M={M} K={K_user}+{K_cand} N={N}")


@pytest.mark.gpu
@pytest.mark.parametrize("N", [64, 256])
@pytest.mark.parametrize("M", [700, 1024, 1100])
def test_many_row_tiles(gpu_lib, M, N):
    """Clusters of six CTAs (M = 700: six row tiles) and eight (M = 1024: eight, the most a
    cluster takes), as three and four CTA pairs at N = 256; no cluster (M = 1100: nine)."""
    cfg = W.LceConfig(name="mt", n_cand=5, n_user=2, M=M, K_user=16, K_cand=80, N=N, seed=M + N)
    check(gpu_lib, W.lce_generate(cfg), f"M={M} N={N}")


@pytest.mark.gpu
def test_no_user_block(gpu_lib):
    cfg = W.LceConfig(name="nu", n_cand=6, n_user=2, M=50, K_user=0, K_cand=40, N=128, seed=4)
    wl = W.lce_generate(cfg)
    Wu, Wc, Xu, Xc, c2u = to_dev(wl)
    out = gpu_lib.lce_fwd(Wu, Wc, Xu, Xc, c2u)
    assert gpu_lib.get_device_error() == 0
    ref = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user)
    assert_close(out.float().cpu().numpy().astype(np.float64), ref, "no user block")


@pytest.mark.gpu
def test_one_candidate_per_user(gpu_lib):
    cfg = W.LceConfig(name="id", n_cand=9, n_user=9, M=70, K_user=24, K_cand=48, N=64, seed=5)
    check(gpu_lib, W.lce_generate(cfg), "identity map")


@pytest.mark.gpu
def test_bad_index_is_reported(gpu_lib):
    wl = W.lce_generate(W.LCE_CONFIGS["lce_tiny_8x3"])
    Wu, Wc, Xu, Xc, c2u = to_dev(wl)
    c2u[5] = 7                                       # outside [0, 3)
    out = torch.full((8, wl.cfg.M, wl.cfg.N), 3.0, dtype=torch.bfloat16, device="cuda")
    gpu_lib.lce_fwd(Wu, Wc, Xu, Xc, c2u, out=out)
    assert gpu_lib.get_device_error() == _lib.IKBO_ERR_INDEX
    assert bool((out[5] == 3.0).all())               # that candidate's rows untouched
    ref = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user, np.array([0, 7]))
    assert_close(out[[0, 7]].float().cpu().numpy().astype(np.float64), ref, "other candidates")
