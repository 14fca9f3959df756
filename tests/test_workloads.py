"""The seeded input generators: determinism, bf16 rounding and the configs' structure."""
import numpy as np
import pytest
import torch

from broadcast_target_attention_gb300 import workloads as W


def test_bf16_rounding_matches_torch():
    rng = np.random.Generator(np.random.PCG64(0))
    x = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    x[:4] = [1.00390625, 1.01171875, -1.00390625, 3.0]   # ties and exact values
    ours = W.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(W.bf16_bits_to_f32(ours),
                          torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_generation_is_deterministic():
    a = W.generate(W.CONFIGS["ratio_1024x15"])
    b = W.generate(W.CONFIGS["ratio_1024x15"])
    for name in ("q", "k", "v", "user_offsets", "cand_to_user"):
        assert np.array_equal(getattr(a, name), getattr(b, name))


def test_headline_structure():
    wl = W.generate(W.CONFIGS["ratio_1024x15"])
    assert wl.n_cand == 1024 and wl.n_user == 15
    assert np.all(wl.counts >= 1) and wl.counts.sum() == 1024
    assert np.all(np.diff(wl.cand_to_user) >= 0)          # sorted
    assert wl.lens.min() >= 256 and wl.lens.max() <= 1024
    assert wl.q.shape == (1024, 4, 1, 128) and wl.k.shape == (wl.T, 4, 128)
    x = W.bf16_bits_to_f32(wl.k)
    assert abs(float(x.std()) - 1.0) < 0.01


def test_odd_group_structure():
    wl = W.generate(W.CONFIGS["odd_groups_2048x16"])
    assert wl.counts.sum() == 2048 and list(wl.counts[-3:]) == [1, 1, 3]
    assert int((wl.counts % 2 == 1).sum()) >= 2
    assert wl.lens.min() >= 64 and wl.lens.max() <= 4096


def test_extreme_and_sweep_structure():
    wl = W.generate(W.CONFIGS["extreme_4096x4"])
    assert wl.counts.sum() == 4096 and wl.n_user == 4
    assert abs(float(W.bf16_bits_to_f32(wl.q).std()) - 0.5) < 0.01
    cfg = W.CONFIGS["sweep_16384x64_d64_lq1"]
    rng = np.random.Generator(np.random.PCG64(cfg.seed))
    counts = W._draw_counts(cfg, rng)
    lens = W._draw_lens(cfg, rng)
    assert counts.sum() == 16384 and lens.min() >= 128 and lens.max() <= 8192


def test_long_user_structure():
    """The long-user set: explicit counts and lengths, as stated; all but the one-user
    counterpart have fewer units than SMs."""
    for name, cfg in W.LONG_CONFIGS.items():
        assert W.attention_config(name) is cfg and name not in W.CONFIGS
        off = np.zeros(cfg.n_user + 1, dtype=np.int64)
        np.cumsum(cfg.lens, out=off[1:])
        c2u = np.repeat(np.arange(cfg.n_user), cfg.counts)
        assert len(c2u) == cfg.n_cand and len(cfg.lens) == cfg.n_user
        cpt = 128 // cfg.Lq
        units = cfg.H * sum(-(-c // cpt) for c in cfg.counts)
        assert (units < 152) == (name != "one_user_10000x700"), name
    wl = W.generate(W.LONG_CONFIGS["few_long_82x4"])
    assert list(np.diff(wl.user_offsets)) == [12000, 3000, 8000, 500]
    assert list(np.bincount(wl.cand_to_user)) == [20, 50, 3, 9]


def test_shuffled_mapping_is_a_permutation():
    wl = W.custom(n_user=3, counts=[4, 2, 5], lens=[3, 4, 5], H=1, D=8, Lq=1, shuffle=True, seed=3)
    assert sorted(wl.cand_to_user.tolist()) == [0] * 4 + [1] * 2 + [2] * 5
    assert np.any(np.diff(wl.cand_to_user) < 0)


@pytest.mark.parametrize("shuffle", [False, True])
def test_hierarchy_structure(shuffle):
    """Every user has at least one vendor and every vendor at least one item; the maps are
    in range, sorted unless shuffled, and the same seed gives the same draw."""
    i2v, v2u, item_user, vpu, ipv = W.draw_hierarchy(1024, 60, 15, seed=51, shuffle=shuffle)
    assert i2v.shape == (1024,) and v2u.shape == (60,) and item_user.shape == (1024,)
    assert vpu.sum() == 60 and ipv.sum() == 1024 and vpu.min() >= 1 and ipv.min() >= 1
    assert np.bincount(v2u, minlength=15).min() >= 1 and np.bincount(i2v, minlength=60).min() >= 1
    assert 0 <= i2v.min() and i2v.max() < 60 and 0 <= v2u.min() and v2u.max() < 15
    assert (np.all(np.diff(i2v) >= 0) and np.all(np.diff(v2u) >= 0)) != shuffle
    again = W.draw_hierarchy(1024, 60, 15, seed=51, shuffle=shuffle)
    assert all(np.array_equal(a, b) for a, b in zip((i2v, v2u, item_user, vpu, ipv), again))
    # uneven at both levels
    assert vpu.max() >= 2 * vpu.min() and ipv.max() >= 4 * ipv.min()
