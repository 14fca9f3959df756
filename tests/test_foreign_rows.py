"""A user's result depends on its own key and value rows only ("In-Kernel Broadcast
Optimization", §3.1: each candidate attends to its own user's sequence).

The last key tile of a user reaches into the rows of the users after it; those keys are
masked, but non-finite values there must not reach the result either (0 x inf is NaN in
P.V).  Here "poison" users without candidates, whose sequences hold +inf, -inf and NaN in
every key and value, sit between the real users and at the end; every kernel, the fused
self + target call and the multi-level call must still match the oracle on every real
candidate (the oracle reads only a user's own rows)."""
import numpy as np
import pytest
import torch

import oracle
from broadcast_target_attention_gb300 import workloads as W
from _helpers import assert_close, out_f64, to_device

pytestmark = pytest.mark.gpu

POS_INF, NEG_INF, NAN = np.uint16(0x7F80), np.uint16(0xFF80), np.uint16(0x7FC0)

# real users (ragged tails: partial 16-key groups, whole groups, a single key, long
# sequences) alternating with poison users (no candidates), one poison user last
REAL_COUNTS = [5, 3, 70, 1, 9, 2]
REAL_LENS = [129, 300, 77, 1, 144, 1000]
POISON_LENS = [37, 5, 200, 1, 16, 90]


def poisoned(D, Lq, seed=31, H=2):
    counts, lens, poison = [], [], []
    for c, L, P in zip(REAL_COUNTS, REAL_LENS, POISON_LENS):
        counts += [c, 0]
        lens += [L, P]
        poison.append(len(lens) - 1)
    wl = W.custom(n_user=len(lens), counts=counts, lens=lens, H=H, D=D, Lq=Lq, seed=seed)
    k, v = wl.k.copy(), wl.v.copy()
    off = wl.user_offsets.astype(np.int64)
    pattern = np.array([POS_INF, NAN, NEG_INF], dtype=np.uint16)
    for u in poison:
        rows = slice(off[u], off[u + 1])
        n = int(off[u + 1] - off[u]) * H * D
        k[rows] = np.resize(pattern, n).reshape(-1, H, D)
        v[rows] = np.resize(pattern[::-1], n).reshape(-1, H, D)
    return W.Workload(cfg=wl.cfg, q=wl.q, k=k, v=v, user_offsets=wl.user_offsets,
                      cand_to_user=wl.cand_to_user, scale=wl.scale), poison


@pytest.mark.parametrize("kernel", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Lq", [1, 3])
def test_foreign_rows_do_not_reach_a_user(gpu_lib, kernel, D, Lq):
    wl, _ = poisoned(D, Lq)
    prev = gpu_lib.set_kernel(kernel)
    try:
        d = to_device(wl)
        out = gpu_lib.attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["cand_to_user"], wl.scale)
        assert gpu_lib.get_device_error() == 0
    finally:
        gpu_lib.set_kernel(prev)
    ref = oracle.attention_wl(wl)
    assert np.all(np.isfinite(ref))
    assert_close(out_f64(out), ref, f"poisoned neighbours kernel={kernel} D={D} Lq={Lq}")


@pytest.mark.parametrize("kernel", [0, 2, 3])
@pytest.mark.parametrize("D", [64, 128])
def test_fused_call_with_poisoned_neighbours(gpu_lib, kernel, D):
    """Target rows of every candidate, and self-attention rows of every real user."""
    wl, poison = poisoned(D, 2)
    qu = W.user_queries(wl)
    prev = gpu_lib.set_kernel(kernel)
    try:
        d = to_device(wl)
        qut = torch.from_numpy(np.ascontiguousarray(qu.view(np.int16))).view(torch.bfloat16).cuda()
        out, out_user = gpu_lib.fused_attn_fwd(d["q"], qut, d["k"], d["v"], d["user_offsets"],
                                               d["cand_to_user"], wl.scale)
        assert gpu_lib.get_device_error() == 0
    finally:
        gpu_lib.set_kernel(prev)
    assert_close(out_f64(out), oracle.attention_wl(wl), f"fused target kernel={kernel} D={D}")
    off = wl.user_offsets.astype(np.int64)
    real_rows = np.concatenate([np.arange(off[u], off[u + 1]) for u in range(len(off) - 1)
                                if u not in poison])
    ref_self = oracle.self_attention(qu, wl.k, wl.v, wl.user_offsets, wl.scale, rows=real_rows)
    got = out_user[torch.as_tensor(real_rows, device=out_user.device)]
    assert_close(out_f64(got), ref_self, f"fused self kernel={kernel} D={D}")


@pytest.mark.parametrize("kernel", [0, 1, 2, 3, 4])
def test_multi_level_call_with_poisoned_neighbours(gpu_lib, kernel):
    """Items reach their user through two maps; the poison users have no vendor."""
    wl, poison = poisoned(128, 1, seed=41)
    real = [u for u in range(wl.n_user) if u not in poison]
    # one vendor per real user, the items (the candidates) keep their order
    vendor_to_user = np.asarray(real, dtype=np.int32)
    vendor_of_user = {u: i for i, u in enumerate(real)}
    item_to_vendor = np.asarray([vendor_of_user[int(u)] for u in wl.cand_to_user], dtype=np.int32)
    prev = gpu_lib.set_kernel(kernel)
    try:
        d = to_device(wl)
        i2v = torch.from_numpy(item_to_vendor).cuda()
        v2u = torch.from_numpy(vendor_to_user).cuda()
        out = gpu_lib.ml_attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], i2v, v2u, wl.scale)
        assert gpu_lib.get_device_error() == 0
    finally:
        gpu_lib.set_kernel(prev)
    ref = oracle.ml_attention(wl.q, wl.k, wl.v, wl.user_offsets, item_to_vendor, vendor_to_user, wl.scale)
    assert_close(out_f64(out), ref, f"multi-level poisoned neighbours kernel={kernel}")
