"""Fused self + target attention ("In-Kernel Broadcast Optimization", §3.3) through the C
ABI: both outputs of one launch against the fp64 oracle, on the named configurations and
on edge cases (ragged and empty sequences, users without candidates, a self-only call,
few units (pair mode), an unsorted map, Lq 1 to 8, D 64 and 128)."""
import numpy as np
import pytest
import torch

import oracle
from broadcast_target_attention_gb300 import _lib
from broadcast_target_attention_gb300 import workloads as W
from _helpers import assert_close, out_f64, to_device

pytestmark = pytest.mark.gpu


def fused(ikbo, wl, qu, kernel=0):
    d = to_device(wl)
    dqu = torch.from_numpy(np.ascontiguousarray(qu).view(np.int16)).view(torch.bfloat16).cuda()
    prev = ikbo.set_kernel(kernel)
    try:
        out, out_user = ikbo.fused_attn_fwd(d["q"], dqu, d["k"], d["v"], d["user_offsets"],
                                            d["cand_to_user"], wl.scale)
        rc = ikbo.get_device_error()
    finally:
        ikbo.set_kernel(prev)
    assert rc == 0, f"device error {rc}"
    return out, out_user


def check(ikbo, wl, what, n_cand_sample=None, n_row_sample=None, kernel=0):
    qu = W.user_queries(wl)
    out, out_user = fused(ikbo, wl, qu, kernel)
    rows = None if n_row_sample is None else W.sample_rows(wl, n_row_sample)
    ref_u = oracle.self_attention(qu, wl.k, wl.v, wl.user_offsets, wl.scale, rows)
    got_u = out_user.float().cpu().numpy().astype(np.float64)
    assert_close(got_u if rows is None else got_u[rows], ref_u, f"{what}: self")
    if wl.n_cand:
        cands = None if n_cand_sample is None else W.sample_candidates(wl, n_cand_sample)
        assert_close(out_f64(out, cands), oracle.attention_wl(wl, cands), f"{what}: target")


@pytest.mark.parametrize("name,n_cand,n_row", [("tiny_8x2", None, None),
                                               ("ratio_1024x15", 256, 256),
                                               ("extreme_4096x4", 64, 192)])
def test_configs(gpu_lib, name, n_cand, n_row):
    check(gpu_lib, W.generate(W.CONFIGS[name]), name, n_cand, n_row)


EDGE = {
    # ragged lengths around the 128-row tile, an empty user, users without candidates
    "ragged": dict(n_user=7, counts=[3, 0, 0, 5, 2, 1, 4], lens=[129, 1, 300, 0, 127, 128, 257]),
    # one user, one candidate, a long sequence: many self tiles, few target tiles
    "long_user": dict(n_user=1, counts=[1], lens=[1500]),
    # few units: clusters of two split each unit's keys (pair mode)
    "pairs": dict(n_user=2, counts=[3, 2], lens=[700, 300]),
    # a last user shorter than a key tile
    "short_last": dict(n_user=4, counts=[4, 3, 2, 5], lens=[300, 170, 90, 20]),
}


@pytest.mark.parametrize("kernel", [2, 3])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Lq", [1, 3, 8])
@pytest.mark.parametrize("case", sorted(EDGE))
def test_edge_cases(gpu_lib, case, Lq, D, kernel):
    """On the one-tile kernel (self tiles of 128 rows) and on the two-tile kernel (self items
    of two 128-row blocks, the second partial or absent)."""
    wl = W.custom(H=2, D=D, Lq=Lq, seed=40 + Lq, **EDGE[case])
    check(gpu_lib, wl, f"{case} Lq={Lq} D={D} kernel={kernel}", kernel=kernel)


@pytest.mark.parametrize("kernel", [2, 3])
def test_unsorted_mapping(gpu_lib, kernel):
    wl = W.custom(n_user=5, counts=[40, 3, 1, 90, 17], lens=[333, 20, 1, 700, 129], H=4, D=128,
                  Lq=2, seed=9, shuffle=True)
    assert np.any(np.diff(wl.cand_to_user) < 0)
    check(gpu_lib, wl, f"unsorted kernel={kernel}", kernel=kernel)


@pytest.mark.parametrize("kernel", [0, 1, 2, 3])
def test_every_kernel_choice(gpu_lib, kernel):
    """The SIMT choice runs on the one-tile kernel; the others as chosen."""
    wl = W.custom(n_user=3, counts=[300, 2, 40], lens=[200, 500, 64], H=2, D=64, Lq=1, seed=12)
    check(gpu_lib, wl, f"kernel choice {kernel}", kernel=kernel)


@pytest.mark.parametrize("kernel", [2, 3])
@pytest.mark.parametrize("D", [64, 128])
def test_self_attention_only(gpu_lib, D, kernel):
    """No candidates: the call computes the user sequence's self-attention alone."""
    base = W.custom(n_user=3, counts=[1, 1, 1], lens=[260, 5, 130], H=2, D=D, Lq=1, seed=6)
    qu = W.user_queries(base)
    d = to_device(base)
    dqu = torch.from_numpy(np.ascontiguousarray(qu).view(np.int16)).view(torch.bfloat16).cuda()
    q0 = d["q"][:0]
    prev = gpu_lib.set_kernel(kernel)
    try:
        out, out_user = gpu_lib.fused_attn_fwd(q0, dqu, d["k"], d["v"], d["user_offsets"],
                                               d["cand_to_user"][:0], base.scale)
    finally:
        gpu_lib.set_kernel(prev)
    assert gpu_lib.get_device_error() == 0
    assert out.shape[0] == 0
    ref = oracle.self_attention(qu, base.k, base.v, base.user_offsets, base.scale)
    assert_close(out_user.float().cpu().numpy().astype(np.float64), ref, "self only")


def test_wrong_row_count_is_reported(gpu_lib):
    """T must equal user_offsets[n_user]: a mismatch is found on the device, nothing written."""
    wl = W.custom(n_user=2, counts=[2, 2], lens=[10, 20], H=2, D=64, Lq=1, seed=1)
    qu = W.user_queries(wl)
    d = to_device(wl)
    k2 = torch.cat([d["k"], d["k"][:4]])          # 34 rows: T stated as 34, offsets end at 30
    v2 = torch.cat([d["v"], d["v"][:4]])
    dqu = torch.cat([torch.from_numpy(qu.view(np.int16)).view(torch.bfloat16).cuda()] * 2)[:34].contiguous()
    out = torch.full_like(d["q"], 7.0)
    out_user = torch.full_like(dqu, 7.0)
    gpu_lib.fused_attn_fwd(d["q"], dqu, k2, v2, d["user_offsets"], d["cand_to_user"], wl.scale,
                           out=out, out_user=out_user)
    assert gpu_lib.get_device_error() == _lib.IKBO_ERR_OFFSETS
    assert bool((out == 7.0).all()) and bool((out_user == 7.0).all())
