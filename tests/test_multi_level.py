"""Multi-level broadcast ("In-Kernel Broadcast Optimization", §5: user -> ads vendor -> ads
item, two nested broadcasts) through the C ABI: target attention and linear compression with
the two maps, against the fp64 multi-level oracle.

CPU: host-side argument checks (nothing reaches the GPU).  GPU: the named configurations,
shuffled maps, every attention kernel (including the planning kernel's walk of the maps
beyond the in-kernel planning limits), empty user sequences, levels without a block, ragged
M, and bad indices at either level."""
import numpy as np
import pytest
import torch

import oracle
from broadcast_target_attention_gb300 import _lib
from broadcast_target_attention_gb300 import build as B
from broadcast_target_attention_gb300 import workloads as W
from _helpers import assert_close, out_f64, to_device


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.lib()


def test_attention_host_checks(lib):
    f = lib.ikbo_ml_attn_fwd
    big = 1 << 40                # a fake, aligned address: every case below is refused before use
    ok = dict(q=big, k=big + (1 << 30), v=big + (2 << 30), off=big, i2v=big, v2u=big, n_item=4,
              n_vendor=3, n_user=2, H=2, Lq=1, D=64, scale=0.125, out=big + (3 << 30))

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["q"], a["k"], a["v"], a["off"], a["i2v"], a["v2u"], a["n_item"], a["n_vendor"],
                 a["n_user"], a["H"], a["Lq"], a["D"], a["scale"], a["out"], None)

    assert call(n_vendor=-1) == _lib.IKBO_ERR_SHAPE
    assert call(D=96) == _lib.IKBO_ERR_SHAPE
    assert call(v2u=None) == _lib.IKBO_ERR_NULL
    assert call(v2u=big + 2) == _lib.IKBO_ERR_ALIGN
    assert call(n_vendor=0) == _lib.IKBO_ERR_INDEX
    assert call(n_item=0, v2u=None) == 0                              # empty batch: no-op
    assert call(out=big) == _lib.IKBO_ERR_ALIAS                        # out over q


def test_lce_host_checks(lib):
    f = lib.ikbo_ml_lce_fwd
    big = 1 << 40
    ok = dict(Wu=big, Wv=big + (1 << 20), Wi=big + (2 << 20), Xu=big + (3 << 20), Xv=big + (4 << 20),
              Xi=big + (5 << 20), i2v=big + (6 << 20), v2u=big + (7 << 20), n_item=6, n_vendor=3,
              n_user=2, M=16, Ku=16, Kv=8, Ki=16, N=64, out=big + (1 << 30))

    def call(**kw):
        a = dict(ok, **kw)
        return f(a["Wu"], a["Wv"], a["Wi"], a["Xu"], a["Xv"], a["Xi"], a["i2v"], a["v2u"], a["n_item"],
                 a["n_vendor"], a["n_user"], a["M"], a["Ku"], a["Kv"], a["Ki"], a["N"], a["out"], None)

    assert call(Kv=12) == _lib.IKBO_ERR_SHAPE
    assert call(Ki=0) == _lib.IKBO_ERR_SHAPE
    assert call(N=320) == _lib.IKBO_ERR_SHAPE
    assert call(n_vendor=-1) == _lib.IKBO_ERR_SHAPE
    assert call(n_item=0) == 0
    assert call(Wv=None) == _lib.IKBO_ERR_NULL
    assert call(v2u=None) == _lib.IKBO_ERR_NULL                        # user block needs it
    assert call(i2v=None) == _lib.IKBO_ERR_NULL
    assert call(n_vendor=0) == _lib.IKBO_ERR_INDEX
    assert call(n_user=0) == _lib.IKBO_ERR_INDEX
    assert call(Xv=big + 8) == _lib.IKBO_ERR_ALIGN
    assert call(i2v=big + 2) == _lib.IKBO_ERR_ALIGN
    assert call(out=ok["Xv"]) == _lib.IKBO_ERR_ALIAS


# ------------------------------------------------------------------------------------ attention

def ml_device(m):
    d = to_device(m.wl)
    d["item_to_vendor"] = torch.from_numpy(m.item_to_vendor).cuda()
    d["vendor_to_user"] = torch.from_numpy(m.vendor_to_user).cuda()
    return d


def run_attn(ikbo, m, kernel=0, d=None):
    d = d or ml_device(m)
    prev = ikbo.set_kernel(kernel)
    try:
        out = ikbo.ml_attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["item_to_vendor"],
                               d["vendor_to_user"], m.wl.scale)
        rc = ikbo.get_device_error()
    finally:
        ikbo.set_kernel(prev)
    return out, rc


def check_attn(ikbo, m, what, n_sample=None, kernel=0):
    out, rc = run_attn(ikbo, m, kernel)
    assert rc == 0, f"{what}: device error {rc}"
    wl = m.wl
    items = None if n_sample is None else W.sample_candidates(wl, n_sample)
    ref = oracle.ml_attention(wl.q, wl.k, wl.v, wl.user_offsets, m.item_to_vendor, m.vendor_to_user,
                              wl.scale, items)
    assert_close(out_f64(out, items), ref, what)


def hand_made(v2u, i2v, lens, H=2, D=64, Lq=1, seed=0):
    """A hierarchy given by its maps; q, k and v drawn as for any workload."""
    v2u = np.asarray(v2u, dtype=np.int32)
    i2v = np.asarray(i2v, dtype=np.int32)
    users = v2u[i2v]                                  # input construction for the test only
    counts = np.bincount(users, minlength=len(lens))
    wl = W.custom(n_user=len(lens), counts=counts.tolist(), lens=list(lens), H=H, D=D, Lq=Lq,
                  seed=seed)
    wl.cand_to_user = users.copy()                    # q row i is item i, in the maps' order
    cfg = W.MlConfig(name="hand", n_item=len(i2v), n_vendor=len(v2u), n_user=len(lens), H=H, D=D,
                     Lq=Lq, seed=seed, len_lo=0, len_hi=0)
    return W.MlWorkload(cfg=cfg, wl=wl, item_to_vendor=i2v, vendor_to_user=v2u)


@pytest.mark.gpu
@pytest.mark.parametrize("name,n_sample", [("ml_tiny_12x5x2", None), ("ml_1024x60x15", 256)])
def test_attention_configs(gpu_lib, name, n_sample):
    check_attn(gpu_lib, W.ml_generate(W.ML_CONFIGS[name]), name, n_sample)


@pytest.mark.gpu
@pytest.mark.parametrize("kernel", [1, 2, 3, 4])
@pytest.mark.parametrize("Lq,D", [(1, 128), (4, 64), (8, 128)])
def test_attention_shuffled_maps_every_kernel(gpu_lib, kernel, Lq, D):
    cfg = W.MlConfig(name="shuf", n_item=700, n_vendor=45, n_user=6, H=2, D=D, Lq=Lq, seed=60 + Lq,
                     len_lo=1, len_hi=700, shuffle=True)
    m = W.ml_generate(cfg)
    assert np.any(np.diff(m.item_to_vendor) < 0) and np.any(np.diff(m.vendor_to_user) < 0)
    check_attn(gpu_lib, m, f"shuffled kernel={kernel} Lq={Lq} D={D}", 160, kernel)


@pytest.mark.gpu
@pytest.mark.parametrize("kernel", [0, 1])
def test_attention_beyond_in_kernel_planning(gpu_lib, kernel):
    """More items than the in-kernel planning takes: the planning kernel walks the maps."""
    cfg = W.MlConfig(name="big", n_item=24000, n_vendor=900, n_user=40, H=1, D=64, Lq=1, seed=61,
                     len_lo=8, len_hi=96, shuffle=True)
    m = W.ml_generate(cfg)
    assert gpu_lib.launches_per_call(cfg.n_item, cfg.n_user) == 2
    check_attn(gpu_lib, m, f"24000 items kernel={kernel}", 192, kernel)


@pytest.mark.gpu
def test_attention_empty_user_and_unreached_vendor(gpu_lib):
    """User 1 has an empty sequence (its items' rows are zero); vendor 4 has no item and a
    user index out of range, which is never read."""
    m = hand_made(v2u=[0, 1, 2, 1, 99], i2v=[0, 0, 1, 2, 3, 2, 0, 1], lens=[130, 0, 257], seed=3)
    out, rc = run_attn(gpu_lib, m)
    assert rc == 0
    wl = m.wl
    m.vendor_to_user = m.vendor_to_user.copy()
    m.vendor_to_user[4] = 0                           # the oracle checks every value; unreached
    ref = oracle.ml_attention(wl.q, wl.k, wl.v, wl.user_offsets, m.item_to_vendor, m.vendor_to_user,
                              wl.scale)
    got = out_f64(out)
    assert_close(got, ref, "empty user")
    assert np.all(got[[2, 4, 7]] == 0)               # items of vendors 1 and 3 (user 1)


@pytest.mark.gpu
@pytest.mark.parametrize("level", ["item_to_vendor", "vendor_to_user"])
def test_attention_bad_index_is_reported(gpu_lib, level):
    m = W.ml_generate(W.ML_CONFIGS["ml_tiny_12x5x2"])
    d = ml_device(m)
    if level == "item_to_vendor":
        d["item_to_vendor"][3] = 5                   # outside [0, 5)
    else:
        d["vendor_to_user"][int(m.item_to_vendor[0])] = -1
    out = torch.full_like(d["q"], 7.0)
    gpu_lib.ml_attn_fwd(d["q"], d["k"], d["v"], d["user_offsets"], d["item_to_vendor"],
                        d["vendor_to_user"], m.wl.scale, out=out)
    assert gpu_lib.get_device_error() == _lib.IKBO_ERR_INDEX
    assert bool((out == 7.0).all())


# ----------------------------------------------------------------------------- linear compression

def lce_device(l):
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).cuda()
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()
    return [bf(l.W_user), bf(l.W_vendor), bf(l.W_item), bf(l.X_user), bf(l.X_vendor), bf(l.X_item),
            i32(l.item_to_vendor), i32(l.vendor_to_user)]


def lce_ref(l, items=None):
    return oracle.ml_lce(l.W_user, l.W_vendor, l.W_item, l.X_user, l.X_vendor, l.X_item,
                         l.item_to_vendor, l.vendor_to_user, items)


def check_lce(ikbo, l, what, items=None):
    out = ikbo.ml_lce_fwd(*lce_device(l))
    assert ikbo.get_device_error() == 0
    got = out.float().cpu().numpy().astype(np.float64)
    if items is not None:
        got = got[items]
    assert_close(got, lce_ref(l, items), what)


def lce_cfg(**kw):
    base = dict(name="s", n_item=23, n_vendor=7, n_user=3, M=130, K_user=24, K_vendor=40, K_item=72,
                N=64, seed=70, shuffle=True)
    base.update(kw)
    return W.lce_ml_generate(W.LceMlConfig(**base))


@pytest.mark.gpu
def test_lce_tiny(gpu_lib):
    check_lce(gpu_lib, W.lce_ml_generate(W.LCE_ML_CONFIGS["lce_ml_tiny_12x5x2"]), "lce_ml_tiny")


@pytest.mark.gpu
def test_lce_pages_sized(gpu_lib):
    l = W.lce_ml_generate(W.LCE_ML_CONFIGS["lce_ml_1024x60x15"])
    items = np.unique(np.concatenate([np.linspace(0, 1023, 40).astype(np.int64),
                                      np.searchsorted(l.item_to_vendor, np.arange(60))]))
    check_lce(gpu_lib, l, "lce_ml_1024x60x15", items)


@pytest.mark.gpu
@pytest.mark.parametrize("N", [64, 192, 256])
@pytest.mark.parametrize("Ku,Kv", [(24, 40), (0, 40), (24, 0), (0, 0)])
def test_lce_levels(gpu_lib, Ku, Kv, N):
    """Every combination of present and absent user and vendor blocks, shuffled maps, ragged M."""
    check_lce(gpu_lib, lce_cfg(K_user=Ku, K_vendor=Kv, N=N, seed=Ku + Kv + N), f"Ku={Ku} Kv={Kv} N={N}")


@pytest.mark.gpu
@pytest.mark.parametrize("M", [1, 700, 1100])
def test_lce_row_tiles(gpu_lib, M):
    """One row, clusters of six CTAs (M = 700) and no cluster (M = 1100) at every level."""
    check_lce(gpu_lib, lce_cfg(M=M, n_item=9, n_vendor=4, n_user=2, K_user=16, K_vendor=8, K_item=80,
                               seed=M), f"M={M}")


@pytest.mark.gpu
@pytest.mark.parametrize("shape", [(5, 5, 5), (6, 6, 2), (8, 2, 2)])
def test_lce_degenerate_ratios(gpu_lib, shape):
    """One vendor per item, one vendor per user with several items, one user per vendor."""
    n_item, n_vendor, n_user = shape
    check_lce(gpu_lib, lce_cfg(n_item=n_item, n_vendor=n_vendor, n_user=n_user, shuffle=False,
                               seed=sum(shape)), f"shape={shape}")


@pytest.mark.gpu
@pytest.mark.parametrize("level", ["item_to_vendor", "vendor_to_user"])
@pytest.mark.parametrize("Kv", [40, 0])
def test_lce_bad_index_is_reported(gpu_lib, level, Kv):
    l = lce_cfg(K_vendor=Kv, shuffle=False)
    args = lce_device(l)
    i2v, v2u = l.item_to_vendor, l.vendor_to_user
    if level == "item_to_vendor":
        args[6][4] = 7                                # outside [0, 7)
        hit = np.array([4])
    else:
        bad_v = int(i2v[10])
        args[7][bad_v] = 3                            # outside [0, 3)
        hit = np.nonzero(i2v == bad_v)[0]
    out = torch.full((l.cfg.n_item, l.cfg.M, l.cfg.N), 3.0, dtype=torch.bfloat16, device="cuda")
    gpu_lib.ml_lce_fwd(*args, out=out)
    assert gpu_lib.get_device_error() == _lib.IKBO_ERR_INDEX
    assert bool((out[torch.as_tensor(hit, device="cuda")] == 3.0).all())   # those items untouched
    rest = np.setdiff1d(np.arange(l.cfg.n_item), hit)
    assert_close(out[torch.as_tensor(rest, device="cuda")].float().cpu().numpy().astype(np.float64),
                 lce_ref(l, rest), "other items")
