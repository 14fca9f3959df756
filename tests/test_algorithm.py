"""The blocked algorithm the CUDA kernel runs, restated in fp64 numpy and held
to the oracle: online softmax over key tiles (with the lazily updated running
maximum) and the split-KV log-sum-exp merge.

Online softmax: "Chapter 4: High-performance Kernels", §4.6.1 (running max m,
running sum l, unnormalised O rescaled by exp(m_prev - m_cur), final O / l).
Split-KV merge: same chapter, §4.6.4 (Flash-Decoding: lse = log Σ exp(lse_c),
o = Σ exp(lse_c - lse) · o_c).
"""
import numpy as np
import pytest

import oracle
from broadcast_target_attention_gb300 import workloads as W

LOG2E = 1.4426950408889634


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def blocked_rows(qrows, K, V, scale, block_n, lazy_threshold):
    """One tile of query rows against one key range, tile by tile, in base 2.

    Returns (o_unnormalised, m, l) with m in log2 units; the running maximum
    is only moved when a tile's maximum exceeds it by more than
    ``lazy_threshold`` (0 = always move), as the kernel does.
    """
    R, D = qrows.shape
    m = np.full(R, -np.inf)
    l = np.zeros(R)
    o = np.zeros((R, D))
    sl2 = scale * LOG2E
    for j0 in range(0, K.shape[0], block_n):
        s = (qrows @ K[j0:j0 + block_n].T) * sl2
        mt = s.max(axis=1)
        move = (mt > m + lazy_threshold) | ~np.isfinite(m)
        m_new = np.where(move, np.maximum(m, mt), m)
        alpha = np.where(np.isfinite(m), np.exp2(m - m_new), 0.0)
        p = np.exp2(s - m_new[:, None])
        l = l * alpha + p.sum(axis=1)
        o = o * alpha[:, None] + p @ V[j0:j0 + block_n]
        m = m_new
    return o, m, l


def merge(parts):
    """Combine (o, m, l) partials of disjoint key ranges (base-2 LSE merge)."""
    M = np.max(np.stack([p[1] for p in parts]), axis=0)
    o = sum(np.exp2(p[1] - M)[:, None] * p[0] for p in parts)
    l = sum(np.exp2(p[1] - M) * p[2] for p in parts)
    return o / l[:, None]


def run_blocked(wl, block_n, lazy, split_keys=None):
    n_cand, H, Lq, D = wl.q.shape
    q, k, v = f64(wl.q), f64(wl.k), f64(wl.v)
    out = np.zeros((n_cand, H, Lq, D))
    off = wl.user_offsets
    for u in range(wl.n_user):
        cands = np.nonzero(wl.cand_to_user == u)[0]
        K, V = k[off[u]:off[u + 1]], v[off[u]:off[u + 1]]
        for h in range(H):
            rows = q[cands, h].reshape(-1, D)          # all candidates of the user share K/V
            if K.shape[0] == 0:
                continue
            if split_keys is None:
                o, m, l = blocked_rows(rows, K[:, h], V[:, h], wl.scale, block_n, lazy)
                res = o / l[:, None]
            else:
                parts = [blocked_rows(rows, K[s:s + split_keys, h], V[s:s + split_keys, h],
                                      wl.scale, block_n, lazy)
                         for s in range(0, K.shape[0], split_keys)]
                res = merge(parts)
            out[cands, h] = res.reshape(len(cands), Lq, D)
    return out


@pytest.mark.parametrize("block_n,lazy", [(128, 0.0), (128, 8.0), (64, 8.0), (16, 0.0)])
def test_online_softmax_matches_one_pass(block_n, lazy):
    wl = W.custom(n_user=3, counts=[5, 1, 4], lens=[300, 7, 129], H=2, D=64, Lq=2, seed=21)
    ref = oracle.attention_wl(wl)
    got = run_blocked(wl, block_n, lazy)
    assert np.max(np.abs(got - ref)) < 1e-12


@pytest.mark.parametrize("split", [128, 256, 100])
def test_split_kv_merge_matches_unsplit(split):
    wl = W.custom(n_user=2, counts=[3, 6], lens=[700, 260], H=2, D=32, Lq=1, seed=22)
    ref = oracle.attention_wl(wl)
    got = run_blocked(wl, 128, 8.0, split_keys=split)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_lazy_max_bounds_the_unnormalised_weights():
    """With threshold 8 (base 2) no weight exceeds 2^8 before normalisation, so
    bf16 P and fp32 row sums stay far from overflow."""
    rng = np.random.Generator(np.random.PCG64(0))
    rows = rng.standard_normal((4, 64)) * 3
    K = rng.standard_normal((512, 64)) * 3
    sl2 = 0.125 * LOG2E
    m = np.full(4, -np.inf)
    worst = 0.0
    for j0 in range(0, 512, 128):
        s = rows @ K[j0:j0 + 128].T * sl2
        mt = s.max(axis=1)
        move = (mt > m + 8.0) | ~np.isfinite(m)
        m = np.where(move, np.maximum(m, mt), m)
        worst = max(worst, float(np.max(np.exp2(s - m[:, None]))))
    assert worst <= 2.0 ** 8
