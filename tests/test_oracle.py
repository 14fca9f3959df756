"""Pins of the CPU fp64 oracle against things other than itself.

Each test fixes the oracle to something the pages or the mathematics
determine: a brute-force restatement on tiny inputs, a library routine on a
special case, closed forms and invariants.  A dropped term, a wrong sign or
index or a transposed operand in the oracle fails at least one of them.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from broadcast_target_attention_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def f64(bits):
    return W.bf16_bits_to_f32(bits).astype(np.float64)


def brute_force(wl):
    """Plain Python floats, indexing the user's K/V directly (no copy)."""
    q = f64(wl.q).tolist()
    k = f64(wl.k).tolist()
    v = f64(wl.v).tolist()
    off = wl.user_offsets.tolist()
    n_cand, H, Lq, D = wl.q.shape
    out = [[[[0.0] * D for _ in range(Lq)] for _ in range(H)] for _ in range(n_cand)]
    for c in range(n_cand):
        u = int(wl.cand_to_user[c])
        for h in range(H):
            for t in range(Lq):
                scores = []
                for j in range(off[u], off[u + 1]):
                    scores.append(wl.scale * math.fsum(q[c][h][t][d] * k[j][h][d] for d in range(D)))
                if not scores:
                    continue
                mx = max(scores)
                e = [math.exp(s - mx) for s in scores]
                z = math.fsum(e)
                for d in range(D):
                    out[c][h][t][d] = math.fsum(e[i] * v[off[u] + i][h][d] for i in range(len(e))) / z
    return np.asarray(out)


def test_tiny_matches_brute_force():
    """Tiny configuration: 2 users, 8 candidates, L = 16 and 24, H=2, D=64, Lq=1."""
    wl = W.generate(W.CONFIGS["tiny_8x2"])
    assert wl.cand_to_user.tolist() == [0, 0, 0, 0, 0, 1, 1, 1]
    assert wl.lens.tolist() == [16, 24]
    got = oracle.attention_wl(wl)
    ref = brute_force(wl)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_multi_token_ragged_matches_brute_force():
    """Several query tokens per candidate, odd groups, lengths 1..9 (incl. an empty user)."""
    wl = W.custom(n_user=5, counts=[3, 1, 2, 1, 2], lens=[9, 1, 0, 5, 7], H=3, D=16, Lq=3, seed=11)
    got = oracle.attention_wl(wl)
    ref = brute_force(wl)
    assert np.max(np.abs(got - ref)) < 1e-12


def test_library_sdpa_special_case():
    """Per user, the candidates' queries against that user's K/V form a dense
    cross-attention, which is what torch's scaled_dot_product_attention
    computes (the GQA-like sharing pattern the IKBO pages compare against)."""
    wl = W.custom(n_user=4, counts=[6, 3, 5, 2], lens=[33, 64, 17, 48], H=4, D=32, Lq=2, seed=5)
    got = oracle.attention_wl(wl)
    q = torch.from_numpy(f64(wl.q))
    k = torch.from_numpy(f64(wl.k))
    v = torch.from_numpy(f64(wl.v))
    c2u = wl.cand_to_user
    off = wl.user_offsets
    for u in range(wl.n_user):
        cands = np.nonzero(c2u == u)[0]
        qu = q[cands]                                   # [r, H, Lq, D]
        qu = qu.permute(1, 0, 2, 3).reshape(wl.cfg.H, -1, wl.cfg.D)   # [H, r*Lq, D]
        ku = k[off[u]:off[u + 1]].permute(1, 0, 2)    # [H, L, D]
        vu = v[off[u]:off[u + 1]].permute(1, 0, 2)
        ref = torch.nn.functional.scaled_dot_product_attention(qu, ku, vu, scale=wl.scale)
        ref = ref.reshape(wl.cfg.H, len(cands), wl.cfg.Lq, wl.cfg.D).permute(1, 0, 2, 3)
        assert np.max(np.abs(got[cands] - ref.numpy())) < 1e-12


def test_broadcast_free_equals_materialised():
    """Indexing the user's K/V through cand_to_user gives bit-for-bit the result
    of first copying K/V once per candidate (IKBO pages, §3.1, Fig. 10)."""
    wl = W.custom(n_user=3, counts=[4, 2, 3], lens=[20, 7, 13], H=2, D=16, Lq=2, seed=3)
    got = oracle.attention_wl(wl)
    off = wl.user_offsets
    kb, vb, offb = [], [], [0]
    for c in range(wl.n_cand):
        u = wl.cand_to_user[c]
        kb.append(wl.k[off[u]:off[u + 1]])
        vb.append(wl.v[off[u]:off[u + 1]])
        offb.append(offb[-1] + off[u + 1] - off[u])
    mat = oracle.attention(wl.q, np.concatenate(kb), np.concatenate(vb), np.asarray(offb),
                           np.arange(wl.n_cand), wl.scale)
    assert np.array_equal(got, mat)


def test_identical_queries_give_identical_rows():
    wl = W.custom(n_user=2, counts=[5, 3], lens=[31, 12], H=2, D=32, Lq=2, seed=4)
    q = wl.q.copy()
    q[1] = q[0]
    q[3] = q[0]
    got = oracle.attention(q, wl.k, wl.v, wl.user_offsets, wl.cand_to_user, wl.scale)
    assert np.array_equal(got[0], got[1]) and np.array_equal(got[0], got[3])
    assert not np.array_equal(got[0], got[2])


def test_length_one_sequence_returns_v():
    wl = W.custom(n_user=3, counts=[2, 3, 1], lens=[5, 1, 4], H=2, D=16, Lq=2, seed=6)
    got = oracle.attention_wl(wl)
    vrow = f64(wl.v[wl.user_offsets[1]])           # [H, D]
    for c in np.nonzero(wl.cand_to_user == 1)[0]:
        for t in range(2):
            assert np.array_equal(got[c, :, t, :], vrow)


def test_weights_are_a_distribution_and_match_scores():
    wl = W.custom(n_user=2, counts=[2, 2], lens=[50, 3], H=2, D=64, Lq=1, seed=7)
    qf, kf = f64(wl.q), f64(wl.k)
    for c in range(wl.n_cand):
        u = wl.cand_to_user[c]
        for h in range(2):
            p = oracle.weights(wl.q, wl.k, wl.user_offsets, wl.cand_to_user, wl.scale, c, h, 0)
            assert np.all(p >= 0) and abs(p.sum() - 1.0) < 1e-12
            s = wl.scale * kf[wl.user_offsets[u]:wl.user_offsets[u + 1], h, :] @ qf[c, h, 0]
            ratio = p / np.exp(s - s.max())          # softmax: p ∝ exp(s)
            assert np.allclose(ratio, ratio[0], rtol=1e-12)


def test_scale_zero_gives_mean_of_user_values():
    wl = W.custom(n_user=3, counts=[2, 2, 2], lens=[8, 3, 6], H=2, D=16, Lq=1, seed=8)
    got = oracle.attention(wl.q, wl.k, wl.v, wl.user_offsets, wl.cand_to_user, 0.0)
    vf = f64(wl.v)
    for c in range(wl.n_cand):
        u = wl.cand_to_user[c]
        mean = vf[wl.user_offsets[u]:wl.user_offsets[u + 1]].mean(axis=0)   # [H, D]
        assert np.max(np.abs(got[c, :, 0, :] - mean)) < 1e-14


def test_candidate_permutation_permutes_rows():
    wl = W.custom(n_user=3, counts=[4, 1, 3], lens=[10, 6, 9], H=2, D=16, Lq=2, seed=9)
    got = oracle.attention_wl(wl)
    perm = np.random.Generator(np.random.PCG64(1)).permutation(wl.n_cand)
    got_p = oracle.attention(wl.q[perm], wl.k, wl.v, wl.user_offsets, wl.cand_to_user[perm], wl.scale)
    assert np.array_equal(got_p, got[perm])


def test_key_order_within_a_user_does_not_matter():
    """Target attention is a set function of the user's history (no mask, no positions)."""
    wl = W.custom(n_user=2, counts=[3, 2], lens=[12, 9], H=2, D=16, Lq=1, seed=10)
    got = oracle.attention_wl(wl)
    k, v = wl.k.copy(), wl.v.copy()
    rows = np.arange(0, 12)[::-1]
    k[0:12], v[0:12] = wl.k[rows], wl.v[rows]
    got2 = oracle.attention(wl.q, k, v, wl.user_offsets, wl.cand_to_user, wl.scale)
    assert np.max(np.abs(got - got2)) < 1e-12


def test_softmax_shift_invariance():
    """Adding one vector w to every key of a user shifts each score row by the
    constant scale·q·w, which softmax ignores.  Dyadic inputs keep K + w exact in bf16."""
    rng = np.random.Generator(np.random.PCG64(2))
    n_cand, H, Lq, D, L = 4, 2, 1, 8, 11
    q = rng.integers(-8, 9, size=(n_cand, H, Lq, D)) / 8.0
    k = rng.integers(-8, 9, size=(L, H, D)) / 8.0
    v = rng.integers(-8, 9, size=(L, H, D)) / 8.0
    w = rng.integers(-4, 5, size=(H, D)) / 4.0
    bf = lambda x: W.f32_to_bf16_bits(x.astype(np.float32))
    off = np.array([0, L])
    c2u = np.zeros(n_cand, dtype=np.int32)
    a = oracle.attention(bf(q), bf(k), bf(v), off, c2u, 0.5)
    b = oracle.attention(bf(q), bf(k + w[None]), bf(v), off, c2u, 0.5)
    assert np.max(np.abs(a - b)) < 1e-12
    k1 = k.copy()
    k1[0] += w          # moving only one key is not a constant shift of the row
    c = oracle.attention(bf(q), bf(k1), bf(v), off, c2u, 0.5)
    assert np.max(np.abs(a - c)) > 1e-6


def test_empty_sequence_gives_zero_rows():
    wl = W.custom(n_user=2, counts=[2, 2], lens=[0, 5], H=1, D=8, Lq=1, seed=12)
    got = oracle.attention_wl(wl)
    assert np.all(got[0:2] == 0.0) and np.any(got[2:] != 0.0)


def test_candidate_subset_matches_full():
    wl = W.generate(W.CONFIGS["ratio_1024x15"])
    sel = W.sample_candidates(wl, 40)
    full = oracle.attention_wl(wl)
    part = oracle.attention_wl(wl, sel)
    assert np.array_equal(part, full[sel])


def test_bad_structure_is_rejected():
    wl = W.custom(n_user=2, counts=[1, 1], lens=[3, 4], H=1, D=8, Lq=1, seed=1)
    with pytest.raises(ValueError):
        oracle.attention(wl.q, wl.k, wl.v, wl.user_offsets, np.array([0, 2]), wl.scale)
    with pytest.raises(ValueError):
        oracle.attention(wl.q, wl.k, wl.v, np.array([0, 5, 4]), wl.cand_to_user, wl.scale)


def test_golden_tiny():
    """Regression pin: values written by tests/golden/make_golden.py from the oracle,
    plus the input bits' digest (same on every machine)."""
    with open(os.path.join(HERE, "golden", "tiny_8x2.json")) as f:
        g = json.load(f)
    wl = W.generate(W.CONFIGS["tiny_8x2"])
    import hashlib
    h = hashlib.sha256(wl.q.tobytes() + wl.k.tobytes() + wl.v.tobytes()).hexdigest()
    assert h == g["inputs_sha256"]
    got = oracle.attention_wl(wl)
    for row in g["rows"]:
        c, hh = row["c"], row["h"]
        assert np.max(np.abs(got[c, hh, 0, :8] - np.asarray(row["out0_8"]))) < 1e-12
