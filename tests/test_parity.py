"""Parity of the CUDA path (through the C ABI) with the fp64 oracle.

Every configuration of the workload table, plus edge cases: ragged tails,
odd and single-candidate groups, empty sequences, users without candidates,
an unsorted candidate map, Lq from 1 to 128, D = 64 and 128, split-KV units.
Tolerance: max-abs 2e-2 and mean-abs 2e-3 for bf16 inputs with fp32
accumulation.  Every GPU kernel is checked: the SIMT kernel (1), the tcgen05
kernel with one query tile per work item (2), the one with two query tiles
of one user and head per item (3) and the one with the key tiles of one query
tile over two softmax warpgroups (4); the full-size configurations also with
the automatic choice (0).
"""
import numpy as np
import pytest
import torch

import oracle
from broadcast_target_attention_gb300 import workloads as W
from _helpers import assert_close, out_f64, to_device

pytestmark = pytest.mark.gpu

KERNELS = [1, 2, 3, 4]
CONFIG_KERNELS = [0, 1, 2, 3, 4]
# (config, number of candidates checked against the oracle; None = all)
CONFIG_SAMPLES = [
    ("tiny_8x2", None),
    ("ratio_1024x15", None),
    ("odd_groups_2048x16", 160),
    ("extreme_4096x4", 96),
    ("sweep_16384x64_d64_lq1", 160),
    ("sweep_16384x64_d64_lq4", 96),
    ("sweep_16384x64_d128_lq1", 160),
    ("sweep_16384x64_d128_lq4", 96),
]

_cache = {}


def workload(name):
    if name not in _cache:
        wl = W.generate(W.attention_config(name))
        _cache.clear()
        _cache[name] = wl
    return _cache[name]


_ref_cache = {}


def config_reference(name, n_sample):
    """(workload, sampled candidates, oracle rows) of a configuration, computed once."""
    if name not in _ref_cache:
        wl = workload(name)
        cands = None if n_sample is None else W.sample_candidates(wl, n_sample)
        _ref_cache.clear()
        _ref_cache[name] = (cands, oracle.attention_wl(wl, cands))
    cands, ref = _ref_cache[name]
    return workload(name), cands, ref


def run(ikbo, wl, kernel, **kw):
    prev = ikbo.set_kernel(kernel)
    try:
        d = to_device(wl)
        out = ikbo.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale, **kw)
        rc = ikbo.get_device_error()
    finally:
        ikbo.set_kernel(prev)
    assert rc == 0, f"device error {rc}"
    return out


@pytest.mark.parametrize("name,n_sample", CONFIG_SAMPLES)
@pytest.mark.parametrize("kernel", CONFIG_KERNELS)
def test_config_matches_oracle(gpu_lib, name, n_sample, kernel):
    wl, cands, ref = config_reference(name, n_sample)
    out = run(gpu_lib, wl, kernel)
    assert_close(out_f64(out, cands), ref, f"{name} kernel={kernel}")
    # properties that hold for every row, checked at full size
    assert torch.isfinite(out.float()).all()


# the long-user set (few units, one much longer than the rest): every kernel choice
LONG_SAMPLES = [(n, 160 if W.LONG_CONFIGS[n].n_cand > 1024 else None) for n in sorted(W.LONG_CONFIGS)]


@pytest.mark.parametrize("name,n_sample", LONG_SAMPLES)
@pytest.mark.parametrize("kernel", CONFIG_KERNELS)
def test_long_user_config_matches_oracle(gpu_lib, name, n_sample, kernel):
    wl, cands, ref = config_reference(name, n_sample)
    out = run(gpu_lib, wl, kernel)
    assert_close(out_f64(out, cands), ref, f"{name} kernel={kernel}")
    assert torch.isfinite(out.float()).all()


EDGE = {
    # ragged tails around the 128-key tile, a length-1 user, an empty user,
    # a user without candidates, odd groups
    "ragged": dict(n_user=7, counts=[3, 1, 0, 5, 2, 1, 4], lens=[129, 1, 300, 0, 127, 128, 257]),
    # one user, one candidate, long sequence: split across CTAs
    "single_long": dict(n_user=1, counts=[1], lens=[5000]),
    # few units, long sequences: the split-KV merge path
    "split": dict(n_user=2, counts=[3, 2], lens=[3001, 1800]),
    # many users with one candidate each (many small units)
    "many_users": dict(n_user=300, counts=[1] * 300, lens=list(range(1, 301))),
    # more candidates than one query tile holds
    "multi_tile": dict(n_user=2, counts=[300, 7], lens=[200, 64]),
    # a last user shorter than a key tile: the tiles of the users before it
    # that reach past the end of k/v
    "short_last": dict(n_user=4, counts=[4, 3, 2, 5], lens=[300, 170, 90, 20]),
    # groups around one and two query tiles (Lq = 1: 128 candidates a tile):
    # full pairs, a pair whose second tile has one candidate, a lone tile,
    # an odd number of tiles
    "tile_pairs": dict(n_user=5, counts=[256, 129, 128, 1, 383], lens=[200, 64, 129, 40, 300]),
}


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Lq", [1, 3, 8])
@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_cases(gpu_lib, case, Lq, D, kernel):
    spec = EDGE[case]
    wl = W.custom(H=2, D=D, Lq=Lq, seed=100 + Lq, **spec)
    out = run(gpu_lib, wl, kernel)
    assert_close(out_f64(out), oracle.attention_wl(wl), f"{case} Lq={Lq} D={D} kernel={kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("D", [64, 128])
def test_output_16_byte_aligned_only(gpu_lib, D, kernel):
    """The output may be 16-byte aligned only (the C ABI's requirement): the epilogues then
    store 16 bytes at a time instead of 32.  Neighbouring bytes stay untouched."""
    wl = W.custom(n_user=4, counts=[130, 3, 1, 140], lens=[200, 1, 300, 129], H=2, D=D, Lq=2, seed=21)
    d = to_device(wl)
    n = d["q"].numel()
    buf = torch.full((n + 16,), 7.0, dtype=torch.bfloat16, device=d["q"].device)
    assert buf.data_ptr() % 32 == 0
    out = buf[8:8 + n].view(d["q"].shape)        # 16 bytes past a 32-byte boundary
    prev = gpu_lib.set_kernel(kernel)
    try:
        gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale, out=out)
        assert gpu_lib.get_device_error() == 0
    finally:
        gpu_lib.set_kernel(prev)
    assert bool((buf[:8] == 7.0).all()) and bool((buf[8 + n:] == 7.0).all())
    assert_close(out_f64(out), oracle.attention_wl(wl), f"16-byte aligned out D={D} kernel={kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("Lq", [5, 64, 128])
def test_large_query_groups(gpu_lib, Lq, kernel):
    wl = W.custom(n_user=3, counts=[5, 2, 9], lens=[140, 70, 390], H=3, D=128, Lq=Lq, seed=7)
    out = run(gpu_lib, wl, kernel)
    assert_close(out_f64(out), oracle.attention_wl(wl), f"Lq={Lq} kernel={kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("D", [64, 128])
def test_unsorted_mapping(gpu_lib, D, kernel):
    wl = W.custom(n_user=5, counts=[40, 3, 1, 90, 17], lens=[333, 20, 1, 700, 129], H=4, D=D, Lq=2,
                  seed=9, shuffle=True)
    assert np.any(np.diff(wl.cand_to_user) < 0)
    out = run(gpu_lib, wl, kernel)
    assert_close(out_f64(out), oracle.attention_wl(wl), f"unsorted D={D} kernel={kernel}")


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("scale", [0.0, -0.125, 1.0, 4.0])
def test_scale_values(gpu_lib, scale, kernel):
    """Any finite scale: 0 gives uniform weights, a negative one reverses the
    order of the scores, large ones move the running maximum tile after tile
    (the rescaling path)."""
    base = W.custom(n_user=3, counts=[70, 5, 33], lens=[900, 129, 300], H=2, D=64, Lq=2, seed=21)
    wl = W.Workload(cfg=base.cfg, q=base.q, k=base.k, v=base.v, user_offsets=base.user_offsets,
                    cand_to_user=base.cand_to_user, scale=scale)
    out = run(gpu_lib, wl, kernel)
    assert_close(out_f64(out), oracle.attention_wl(wl), f"scale={scale} kernel={kernel}")


def test_kernels_agree_at_full_size(gpu_lib):
    wl = workload("odd_groups_2048x16")
    a = run(gpu_lib, wl, 1).float()
    for kernel in (2, 3, 4):
        b = run(gpu_lib, wl, kernel).float()
        assert (a - b).abs().max().item() <= 2e-2, kernel


@pytest.mark.parametrize("name", ["ratio_1024x15", "extreme_4096x4"])
def test_identical_queries_give_identical_rows(gpu_lib, name):
    """A property at any size: candidates of one user with the same queries get the same
    rows (for the second configuration across the 64 query tiles of its largest user, run
    two tiles per work item)."""
    wl = workload(name)
    q = wl.q.copy()
    user = 3 if name == "ratio_1024x15" else int(np.bincount(wl.cand_to_user).argmax())
    first = np.nonzero(wl.cand_to_user == user)[0]
    q[first[1:]] = q[first[0]]
    wl2 = W.Workload(cfg=wl.cfg, q=q, k=wl.k, v=wl.v, user_offsets=wl.user_offsets,
                     cand_to_user=wl.cand_to_user, scale=wl.scale)
    out = run(gpu_lib, wl2, 0)
    rows = out[torch.as_tensor(first, device=out.device)]
    assert torch.equal(rows, rows[:1].expand_as(rows))


def test_empty_batch_is_a_noop(gpu_lib):
    wl = W.custom(n_user=2, counts=[1, 1], lens=[3, 3], H=1, D=64, Lq=1)
    d = to_device(wl)
    q = d["q"][:0]
    out = gpu_lib.attn_fwd(q, d["k"], d["v"], d["user_offsets"], d["cand_to_user"][:0], 0.1)
    assert out.shape[0] == 0


@pytest.mark.parametrize("name", ["ratio_1024x15", "extreme_4096x4"])
def test_repeated_calls_are_deterministic(gpu_lib, name):
    wl = workload(name)
    a = run(gpu_lib, wl, 0)
    b = run(gpu_lib, wl, 0)
    assert torch.equal(a, b)


@pytest.mark.parametrize("kernel", KERNELS)
@pytest.mark.parametrize("sharp", [1.0, 4.0])
def test_very_long_sequence(gpu_lib, kernel, sharp):
    """One user with 65,000 keys (508 key tiles, split over a cluster pair or planned apart):
    the running maximum and the lazy rescale over hundreds of tiles.  A scale 4x the usual
    one makes the weights peakier and the maximum move more often (inputs and outputs stay
    of unit scale, the regime of the tolerance)."""
    wl = W.custom(n_user=2, counts=[5, 2], lens=[65000, 300], H=2, D=128, Lq=3, seed=77)
    scale = wl.scale * sharp
    prev = gpu_lib.set_kernel(kernel)
    try:
        d = to_device(wl)
        out = gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], scale)
        assert gpu_lib.get_device_error() == 0
    finally:
        gpu_lib.set_kernel(prev)
    ref = oracle.attention(wl.q, wl.k, wl.v, wl.user_offsets, wl.cand_to_user, scale)
    assert_close(out_f64(out), ref, f"65k keys kernel={kernel} scale x{sharp}")
