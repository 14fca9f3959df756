"""Pins of the oracle's self-attention of the user sequence ("In-Kernel Broadcast
Optimization", §3.3: queries from the user side, the same keys and values as the target
attention, full attention without a causal mask) against things other than itself."""
import math

import numpy as np
import torch

import oracle
from broadcast_target_attention_gb300 import workloads as W


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def brute_force_self(qu, k, v, off, scale):
    """Plain Python floats: every row of user u against all of user u's keys."""
    q = f64(qu).tolist()
    kk = f64(k).tolist()
    vv = f64(v).tolist()
    T, H, D = qu.shape
    out = [[[0.0] * D for _ in range(H)] for _ in range(T)]
    for u in range(len(off) - 1):
        for r in range(off[u], off[u + 1]):
            for h in range(H):
                s = [scale * math.fsum(q[r][h][d] * kk[j][h][d] for d in range(D))
                     for j in range(off[u], off[u + 1])]
                m = max(s)
                e = [math.exp(x - m) for x in s]
                tot = math.fsum(e)
                for d in range(D):
                    out[r][h][d] = math.fsum(e[i] * vv[off[u] + i][h][d] for i in range(len(e))) / tot
    return np.asarray(out)


def tiny(lens=(5, 1, 0, 7), H=2, D=8, seed=11):
    wl = W.custom(n_user=len(lens), counts=[1] * len(lens), lens=list(lens), H=H, D=D, Lq=1, seed=seed)
    return wl, W.user_queries(wl)


def test_matches_brute_force():
    wl, qu = tiny()
    got = oracle.self_attention(qu, wl.k, wl.v, wl.user_offsets, wl.scale)
    ref = brute_force_self(qu, wl.k, wl.v, wl.user_offsets.tolist(), wl.scale)
    assert np.abs(got - ref).max() < 1e-12


def test_library_sdpa_on_one_dense_user():
    """One user: plain dense self-attention, which torch's fp64 SDPA computes (non-causal)."""
    wl, qu = tiny(lens=(37,), H=3, D=16, seed=5)
    got = oracle.self_attention(qu, wl.k, wl.v, wl.user_offsets, wl.scale)
    t = lambda a: torch.from_numpy(f64(a)).permute(1, 0, 2).unsqueeze(0)   # [1, H, L, D]
    ref = torch.nn.functional.scaled_dot_product_attention(t(qu), t(wl.k), t(wl.v), is_causal=False,
                                                           scale=wl.scale)
    ref = ref.squeeze(0).permute(1, 0, 2).numpy()
    assert np.abs(got - ref).max() < 1e-12


def test_rows_attend_to_their_own_user_only():
    """Changing another user's keys and values leaves a user's rows unchanged."""
    wl, qu = tiny(lens=(6, 9), seed=3)
    a = oracle.self_attention(qu, wl.k, wl.v, wl.user_offsets, wl.scale)
    k2, v2 = wl.k.copy(), wl.v.copy()
    k2[6:] = W.f32_to_bf16_bits(np.full(k2[6:].shape, 3.0, np.float32))
    v2[6:] = W.f32_to_bf16_bits(np.full(v2[6:].shape, -2.0, np.float32))
    b = oracle.self_attention(qu, k2, v2, wl.user_offsets, wl.scale)
    assert np.array_equal(a[:6], b[:6])
    assert not np.allclose(a[6:], b[6:])
    assert np.allclose(b[6:], -2.0, atol=1e-12)       # every weight on a value row of -2


def test_length_one_user_returns_its_value_row():
    wl, qu = tiny(lens=(4, 1, 3), seed=8)
    got = oracle.self_attention(qu, wl.k, wl.v, wl.user_offsets, wl.scale)
    assert np.array_equal(got[4], f64(wl.v[4]))


def test_scale_zero_gives_mean_of_user_values():
    wl, qu = tiny(lens=(5, 3), seed=2)
    got = oracle.self_attention(qu, wl.k, wl.v, wl.user_offsets, 0.0)
    v = f64(wl.v)
    assert np.abs(got[:5] - v[:5].mean(axis=0)).max() < 1e-12
    assert np.abs(got[5:] - v[5:].mean(axis=0)).max() < 1e-12


def test_equals_target_attention_with_each_row_as_a_candidate():
    """A self-attention row is a one-token candidate of its own user ([IKBO] §3.3: only the
    query source differs): compare with the target attention of that mapping."""
    wl, qu = tiny(lens=(5, 1, 0, 7), seed=13)
    T, H, D = qu.shape
    c2u = np.repeat(np.arange(4, dtype=np.int32), np.diff(wl.user_offsets))
    tgt = oracle.attention(qu.reshape(T, H, 1, D), wl.k, wl.v, wl.user_offsets, c2u, wl.scale)
    got = oracle.self_attention(qu, wl.k, wl.v, wl.user_offsets, wl.scale)
    assert np.abs(got - tgt[:, :, 0, :]).max() < 1e-12


def test_row_subset_matches_full():
    wl, qu = tiny(lens=(9, 4, 11), seed=4)
    full = oracle.self_attention(qu, wl.k, wl.v, wl.user_offsets, wl.scale)
    rows = np.array([0, 8, 9, 12, 13, 23], dtype=np.int64)
    sub = oracle.self_attention(qu, wl.k, wl.v, wl.user_offsets, wl.scale, rows)
    assert np.array_equal(sub, full[rows])
