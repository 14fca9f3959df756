"""Pins of the multi-level oracle ("In-Kernel Broadcast Optimization", §5: user -> ads vendor
-> ads item, two nested broadcasts) against things other than itself: a top-down walk of the
drawn hierarchy with plain-float attention, the materialised two-level broadcast through
torch's fp64 SDPA, the reductions to the two-level oracles when a level is trivial, the
library's batched product on identity maps, and the decomposition of the linear compression
into three per-level products."""
import math

import numpy as np
import pytest
import torch

import oracle
from oracle import multi_level
from broadcast_target_attention_gb300 import workloads as W


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def small(shuffle=False, n_item=14, n_vendor=6, n_user=3, seed=7, Lq=2):
    return W.ml_generate(W.MlConfig(name="s", n_item=n_item, n_vendor=n_vendor, n_user=n_user, H=2,
                                    D=8, Lq=Lq, seed=seed, len_lo=1, len_hi=9, shuffle=shuffle))


@pytest.mark.parametrize("shuffle", [False, True])
def test_walk_matches_the_drawn_structure(shuffle):
    m = small(shuffle, n_item=300, n_vendor=40, n_user=7)
    users = multi_level.walk(m.item_to_vendor, m.vendor_to_user, 7)
    assert np.array_equal(users, m.wl.cand_to_user)
    if shuffle:
        assert np.any(np.diff(m.item_to_vendor) < 0) and np.any(np.diff(m.vendor_to_user) < 0)


@pytest.mark.parametrize("shuffle", [False, True])
def test_attention_against_a_top_down_walk(shuffle):
    """Users, then each user's vendors, then each vendor's items; plain Python floats."""
    m = small(shuffle)
    wl = m.wl
    q, k, v = (f64(x).tolist() for x in (wl.q, wl.k, wl.v))
    off = wl.user_offsets.tolist()
    n_item, H, Lq, D = wl.q.shape
    ref = np.full((n_item, H, Lq, D), np.nan)
    for u in range(wl.n_user):
        for vd in [j for j in range(len(m.vendor_to_user)) if m.vendor_to_user[j] == u]:
            for i in [j for j in range(n_item) if m.item_to_vendor[j] == vd]:
                for h in range(H):
                    for t in range(Lq):
                        s = [wl.scale * math.fsum(q[i][h][t][d] * k[r][h][d] for d in range(D))
                             for r in range(off[u], off[u + 1])]
                        mx = max(s)
                        e = [math.exp(x - mx) for x in s]
                        tot = math.fsum(e)
                        for d in range(D):
                            ref[i, h, t, d] = math.fsum(e[j] * v[off[u] + j][h][d]
                                                        for j in range(len(e))) / tot
    assert not np.isnan(ref).any()                   # every item reached exactly once
    got = oracle.ml_attention(wl.q, wl.k, wl.v, wl.user_offsets, m.item_to_vendor, m.vendor_to_user,
                              wl.scale)
    assert np.abs(got - ref).max() < 1e-12


def test_attention_against_the_materialised_broadcast():
    """The form IKBO removes: every vendor gets its own copy of its user's keys and values,
    every item its own copy of its vendor's; then dense attention per item (torch fp64
    SDPA, non-causal)."""
    m = small(True, seed=9)
    wl = m.wl
    off = wl.user_offsets
    kf, vf, qf = f64(wl.k), f64(wl.v), f64(wl.q)
    vendor_kv = [(kf[off[u]:off[u + 1]].copy(), vf[off[u]:off[u + 1]].copy()) for u in m.vendor_to_user]
    got = oracle.ml_attention(wl.q, wl.k, wl.v, off, m.item_to_vendor, m.vendor_to_user, wl.scale)
    for i, vd in enumerate(m.item_to_vendor):
        ki, vi = (x.copy() for x in vendor_kv[vd])
        t = lambda a: torch.from_numpy(a).permute(1, 0, 2).unsqueeze(0)   # [1, H, L, D]
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(qf[i]).unsqueeze(0), t(ki), t(vi), scale=wl.scale).squeeze(0).numpy()
        assert np.abs(got[i] - ref).max() < 1e-12


def test_one_vendor_per_user_is_the_two_level_attention():
    m = small(n_item=10, n_vendor=3, n_user=3, seed=4)
    assert np.array_equal(m.vendor_to_user, np.arange(3))
    wl = m.wl
    got = oracle.ml_attention(wl.q, wl.k, wl.v, wl.user_offsets, m.item_to_vendor, m.vendor_to_user,
                              wl.scale)
    ref = oracle.attention(wl.q, wl.k, wl.v, wl.user_offsets, m.item_to_vendor, wl.scale)
    assert np.array_equal(got, ref)


def test_one_item_per_vendor_is_the_two_level_attention():
    m = small(n_item=6, n_vendor=6, n_user=2, seed=5)
    assert np.array_equal(m.item_to_vendor, np.arange(6))
    wl = m.wl
    got = oracle.ml_attention(wl.q, wl.k, wl.v, wl.user_offsets, m.item_to_vendor, m.vendor_to_user,
                              wl.scale)
    ref = oracle.attention(wl.q, wl.k, wl.v, wl.user_offsets, m.vendor_to_user, wl.scale)
    assert np.array_equal(got, ref)


def test_item_subset_matches_full():
    m = small(True)
    wl = m.wl
    a = (wl.q, wl.k, wl.v, wl.user_offsets, m.item_to_vendor, m.vendor_to_user, wl.scale)
    full = oracle.ml_attention(*a)
    sel = np.array([0, 5, 13], dtype=np.int64)
    assert np.array_equal(oracle.ml_attention(*a, items=sel), full[sel])


def test_out_of_range_maps_raise():
    m = small()
    wl = m.wl
    bad_v = m.item_to_vendor.copy()
    bad_v[3] = len(m.vendor_to_user)
    with pytest.raises(ValueError):
        oracle.ml_attention(wl.q, wl.k, wl.v, wl.user_offsets, bad_v, m.vendor_to_user, wl.scale)
    bad_u = m.vendor_to_user.copy()
    bad_u[0] = -1
    with pytest.raises(ValueError):
        oracle.ml_attention(wl.q, wl.k, wl.v, wl.user_offsets, m.item_to_vendor, bad_u, wl.scale)


# ---------------------------------------------------------------------------- linear compression

def lce_small(K_user=13, K_vendor=9, K_item=21, shuffle=True, seed=52, n_item=12, n_vendor=5,
              n_user=2, M=11, N=64):
    return W.lce_ml_generate(W.LceMlConfig(name="s", n_item=n_item, n_vendor=n_vendor, n_user=n_user,
                                           M=M, K_user=K_user, K_vendor=K_vendor, K_item=K_item,
                                           N=N, seed=seed, shuffle=shuffle))


def lce_args(l):
    return (l.W_user, l.W_vendor, l.W_item, l.X_user, l.X_vendor, l.X_item, l.item_to_vendor,
            l.vendor_to_user)


def test_lce_brute_force():
    l = lce_small(M=5)
    got = oracle.ml_lce(*lce_args(l))
    Wu, Wv, Wi, Xu, Xv, Xi = (f64(x).tolist() for x in lce_args(l)[:6])
    for i in range(len(Xi)):
        u, vd = int(l.item_user[i]), int(l.item_to_vendor[i])
        for m_ in range(len(Wu)):
            for n in range(len(Xi[0][0])):
                ref = math.fsum([Wu[m_][k] * Xu[u][k][n] for k in range(len(Wu[0]))] +
                                [Wv[m_][k] * Xv[vd][k][n] for k in range(len(Wv[0]))] +
                                [Wi[m_][k] * Xi[i][k][n] for k in range(len(Wi[0]))])
                assert abs(got[i, m_, n] - ref) < 1e-12


def test_lce_decomposes_into_three_products():
    """§2.1 at both levels: each block's product computed at its own batch size, then
    gathered through the drawn structure."""
    l = lce_small()
    got = oracle.ml_lce(*lce_args(l))
    user = np.einsum("mk,ukn->umn", f64(l.W_user), f64(l.X_user))
    vendor = np.einsum("mk,vkn->vmn", f64(l.W_vendor), f64(l.X_vendor))
    item = np.einsum("mk,ikn->imn", f64(l.W_item), f64(l.X_item))
    ref = user[l.item_user] + vendor[l.item_to_vendor] + item
    assert np.abs(got - ref).max() < 1e-12


def test_lce_without_a_vendor_block_is_the_two_level_lce():
    l = lce_small(K_vendor=0)
    got = oracle.ml_lce(*lce_args(l))
    ref = oracle.lce(l.W_user, l.W_item, l.X_user, l.X_item, l.item_user)
    assert np.array_equal(got, ref)


def test_lce_without_a_user_block_is_the_two_level_lce_over_vendors():
    l = lce_small(K_user=0)
    got = oracle.ml_lce(*lce_args(l))
    ref = oracle.lce(l.W_vendor, l.W_item, l.X_vendor, l.X_item, l.item_to_vendor)
    assert np.array_equal(got, ref)


def test_lce_identity_maps_are_the_plain_batched_product():
    l = lce_small(n_item=4, n_vendor=4, n_user=4, shuffle=False, M=9, N=64)
    assert np.array_equal(l.item_to_vendor, np.arange(4)) and np.array_equal(l.vendor_to_user, np.arange(4))
    got = oracle.ml_lce(*lce_args(l))
    Wt = torch.from_numpy(np.concatenate([f64(l.W_user), f64(l.W_vendor), f64(l.W_item)], axis=1))
    Xt = torch.from_numpy(np.concatenate([f64(l.X_user), f64(l.X_vendor), f64(l.X_item)], axis=1))
    assert np.abs(got - torch.matmul(Wt, Xt).numpy()).max() < 1e-12


def test_lce_same_vendor_same_item_block_same_output():
    l = lce_small(shuffle=False)
    Xi = l.X_item.copy()
    a, b = [i for i in range(12) if l.item_to_vendor[i] == l.item_to_vendor[0]][:2]
    Xi[b] = Xi[a]
    args = list(lce_args(l))
    args[5] = Xi
    got = oracle.ml_lce(*args)
    assert np.array_equal(got[a], got[b])
    # another vendor of the same user: the vendor term differs
    c = next(i for i in range(12) if l.item_to_vendor[i] != l.item_to_vendor[a]
             and l.item_user[i] == l.item_user[a])
    Xi[c] = Xi[a]
    got = oracle.ml_lce(*args[:5], Xi, *args[6:])
    assert not np.allclose(got[c], got[a])
