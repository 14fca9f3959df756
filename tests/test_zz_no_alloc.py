"""The allocation-free entry point, ikbo_attn_fwd_noalloc, called through the C ABI.

It is meant for callers whose memory manager owns all device memory (or that
run without stream-ordered memory pools) and so cannot let the library
allocate: its scratch is a fixed array inside the library.  It must give the
result of ikbo_attn_fwd, and of the oracle, call after call, since every call
reuses the same array; and it must leave every memory pool untouched.  This
file is collected last on purpose.
"""
import ctypes

import pytest
import torch

import oracle
from broadcast_target_attention_gb300 import _lib
from broadcast_target_attention_gb300 import workloads as W
from _helpers import MAX_ABS, MEAN_ABS, assert_close, out_f64, to_device

pytestmark = pytest.mark.gpu


def _call(fn, d, wl, out):
    n_cand, H, Lq, D = d["q"].shape
    rc = fn(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["user_offsets"].data_ptr(),
            d["cand_to_user"].data_ptr(), n_cand, wl.n_user, H, Lq, D, ctypes.c_float(wl.scale),
            out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return rc


class _DefaultPool:
    """The current device's default stream-ordered pool, read through the driver API."""
    USED_MEM_HIGH, RESERVED_MEM_CURRENT, RELEASE_THRESHOLD = 8, 5, 4

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def get(self, attr):
        v = ctypes.c_uint64()
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
        return v.value

    def snapshot(self):
        return {a: self.get(a) for a in (self.USED_MEM_HIGH, self.RESERVED_MEM_CURRENT,
                                         self.RELEASE_THRESHOLD)}


def _library_pool(reset=False):
    now, high = ctypes.c_uint64(), ctypes.c_uint64()
    assert _lib.lib().ikbo_pool_usage(1 if reset else 0, ctypes.byref(now), ctypes.byref(high)) == 0
    return now.value, high.value


@pytest.mark.parametrize("name", ["ratio_1024x15", "odd_groups_2048x16"])
def test_noalloc_matches_attn_fwd_on_two_calls_in_a_row(gpu_lib, name):
    lib = _lib.lib()
    wl = W.generate(W.CONFIGS[name])
    cands = None if wl.n_cand <= 1024 else W.sample_candidates(wl, 160)
    ref_oracle = oracle.attention_wl(wl, cands)
    d = to_device(wl)
    ref = torch.empty_like(d["q"])
    assert _call(lib.ikbo_attn_fwd, d, wl, ref) == 0
    assert lib.ikbo_get_device_error(None) == 0
    for _ in range(2):
        out = torch.full_like(d["q"], 3.0)
        assert _call(lib.ikbo_attn_fwd_noalloc, d, wl, out) == 0
        assert lib.ikbo_get_device_error(None) == 0
        diff = (out.float() - ref.float()).abs()
        assert diff.max().item() <= MAX_ABS and diff.mean().item() <= MEAN_ABS
        assert_close(out_f64(out, cands), ref_oracle, f"noalloc {name}")


def test_noalloc_second_call_does_not_depend_on_the_first(gpu_lib):
    """A different, smaller problem right after a large one reuses the array."""
    lib = _lib.lib()
    big = W.generate(W.CONFIGS["ratio_1024x15"])
    small = W.custom(n_user=3, counts=[5, 1, 2], lens=[300, 17, 129], H=2, D=64, Lq=3, seed=4)
    for wl in (big, small):
        d = to_device(wl)
        ref = torch.empty_like(d["q"])
        out = torch.empty_like(d["q"])
        assert _call(lib.ikbo_attn_fwd, d, wl, ref) == 0
        assert _call(lib.ikbo_attn_fwd_noalloc, d, wl, out) == 0
        assert lib.ikbo_get_device_error(None) == 0
        diff = (out.float() - ref.float()).abs()
        assert diff.max().item() <= MAX_ABS and diff.mean().item() <= MEAN_ABS
        assert_close(out_f64(out), oracle.attention_wl(wl), "noalloc after a larger call")


def test_noalloc_leaves_every_pool_untouched(gpu_lib):
    """No allocation from the library's pool or the device's default pool, and no pool
    attribute changed, over several calls (a regression to a pool allocation would raise
    a high-water mark)."""
    lib = _lib.lib()
    wl = W.generate(W.CONFIGS["ratio_1024x15"])
    d = to_device(wl)
    out = torch.empty_like(d["q"])
    assert _call(lib.ikbo_attn_fwd_noalloc, d, wl, out) == 0      # first call: set-up
    torch.cuda.synchronize()
    default = _DefaultPool()
    before = default.snapshot()
    used_now, _ = _library_pool(reset=True)
    for _ in range(4):
        assert _call(lib.ikbo_attn_fwd_noalloc, d, wl, out) == 0
    assert lib.ikbo_get_device_error(None) == 0
    torch.cuda.synchronize()
    assert default.snapshot() == before
    now, high = _library_pool()
    assert now == used_now and high <= used_now


def _minimal(n_cand, n_user, H, Lq, D):
    """Device tensors of a configuration's sizes: every user one key, candidates sorted."""
    dev = torch.device("cuda")
    q = torch.zeros(n_cand, H, Lq, D, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(n_user, H, D, dtype=torch.bfloat16, device=dev)
    off = torch.arange(n_user + 1, dtype=torch.int32, device=dev)
    c2u = (torch.arange(n_cand, device=dev) * n_user // n_cand).to(torch.int32)
    return dict(q=q, k=k, v=k.clone(), user_offsets=off, cand_to_user=c2u)


@pytest.mark.parametrize("name", sorted(W.CONFIGS) + sorted(W.LONG_CONFIGS))
def test_noalloc_fits_every_configuration_and_kernel(gpu_lib, name):
    """The fixed array holds the scratch of every configuration's sizes with every kernel
    choice (the need depends on the sizes and the kernel, not on the values)."""
    lib = _lib.lib()
    cfg = W.attention_config(name)
    d = _minimal(cfg.n_cand, cfg.n_user, cfg.H, cfg.Lq, cfg.D)
    out = torch.empty_like(d["q"])
    wl = type("Sizes", (), {"n_user": cfg.n_user, "scale": cfg.D ** -0.5})
    for kernel in (0, 1, 2, 3, 4):
        prev = lib.ikbo_set_kernel(kernel)
        try:
            assert _call(lib.ikbo_attn_fwd_noalloc, d, wl, out) == 0, (name, kernel)
            assert lib.ikbo_get_device_error(None) == 0, (name, kernel)
        finally:
            lib.ikbo_set_kernel(prev)
        # every key is 0 and every value 0, one key per user: the output is 0
        assert torch.count_nonzero(out).item() == 0, (name, kernel)


def test_noalloc_rejects_a_call_that_needs_more_scratch(gpu_lib):
    """Many heads times many query tiles overflow the fixed array: refused, nothing run."""
    lib = _lib.lib()
    n_cand, n_user, H, Lq, D = 1 << 20, 1 << 20, 64, 128, 128
    A = 1 << 20
    # fake, never dereferenced addresses; out placed past the end of q
    rc = lib.ikbo_attn_fwd_noalloc(A, 2 * A, 3 * A, 4 * A, 5 * A, n_cand, n_user, H, Lq, D,
                                   ctypes.c_float(0.1), 1 << 44, None)
    assert rc == _lib.IKBO_ERR_SCRATCH
