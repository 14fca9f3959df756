"""Pins of the linear-compression oracle ("In-Kernel Broadcast Optimization", §2) against
things other than itself: brute force on tiny inputs, the library's batched product on the
identity mapping, the decomposition the pages prove exact (§2.1), zero padding of K (§2.2,
proof 1) and the broadcast invariants."""
import math

import numpy as np
import torch

import oracle
from broadcast_target_attention_gb300 import workloads as W


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def tiny():
    return W.lce_generate(W.LCE_CONFIGS["lce_tiny_8x3"])


def test_matches_brute_force():
    wl = tiny()
    got = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user)
    Wu, Wc, Xu, Xc = (f64(x).tolist() for x in (wl.W_user, wl.W_cand, wl.X_user, wl.X_cand))
    M, N = len(Wu), len(Xc[0][0])
    for b in range(len(Xc)):
        u = int(wl.cand_to_user[b])
        for m in range(M):
            for n in range(N):
                ref = math.fsum([Wu[m][k] * Xu[u][k][n] for k in range(len(Wu[0]))] +
                                [Wc[m][k] * Xc[b][k][n] for k in range(len(Wc[0]))])
                assert abs(got[b, m, n] - ref) < 1e-12


def test_identity_mapping_is_the_plain_batched_product():
    """Every candidate its own user: the batched (M, K) @ (B, K, N) product of the pages'
    baseline, which torch computes in fp64."""
    cfg = W.LceConfig(name="id", n_cand=5, n_user=5, M=19, K_user=8, K_cand=16, N=64, seed=3)
    wl = W.lce_generate(cfg)
    got = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user)
    Wt = torch.from_numpy(np.concatenate([f64(wl.W_user), f64(wl.W_cand)], axis=1))
    Xt = torch.from_numpy(np.concatenate([f64(wl.X_user)[wl.cand_to_user], f64(wl.X_cand)], axis=1))
    ref = torch.matmul(Wt, Xt).numpy()
    assert np.abs(got - ref).max() < 1e-12


def test_decomposition_is_exact():
    """§2.1: W @ [X_user ; X_cand] = W_user @ X_user + W_cand @ X_cand."""
    wl = tiny()
    got = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user)
    user = np.einsum("mk,ukn->umn", f64(wl.W_user), f64(wl.X_user))
    cand = np.einsum("mk,bkn->bmn", f64(wl.W_cand), f64(wl.X_cand))
    assert np.abs(got - (user[wl.cand_to_user] + cand)).max() < 1e-12


def test_zero_padding_of_k_is_exact():
    """§2.2, proof 1: the zero columns / rows that round K up to a multiple of 8 change nothing."""
    wl = tiny()
    c = wl.cfg
    full = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user)
    bare = oracle.lce(wl.W_user[:, :c.K_user], wl.W_cand[:, :c.K_cand], wl.X_user[:, :c.K_user],
                      wl.X_cand[:, :c.K_cand], wl.cand_to_user)
    assert np.array_equal(full, bare)


def test_same_user_same_candidate_block_same_output():
    wl = tiny()
    Xc = wl.X_cand.copy()
    Xc[3] = Xc[2]                               # candidates 2 and 3 both belong to user 1
    assert wl.cand_to_user[2] == wl.cand_to_user[3]
    got = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, Xc, wl.cand_to_user)
    assert np.array_equal(got[2], got[3])
    Xc[5] = Xc[2]                               # candidate 5 belongs to user 2: differs
    got = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, Xc, wl.cand_to_user)
    assert not np.allclose(got[5], got[2])


def test_candidate_subset_matches_full():
    wl = tiny()
    full = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user)
    sel = np.array([0, 4, 7], dtype=np.int64)
    sub = oracle.lce(wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user, sel)
    assert np.array_equal(sub, full[sel])
