"""The allocation-free entry point, ikbo_attn_fwd_noalloc, called through the C ABI.

It is meant for callers whose memory manager owns all device memory (or that
run without stream-ordered memory pools) and so cannot let the library
allocate: its scratch is a fixed array inside the library.  It must give the
same result as ikbo_attn_fwd, call after call, since every call reuses the
same array.  This file is collected last on purpose.
"""
import ctypes

import pytest
import torch

from broadcast_target_attention_gb300 import _lib
from broadcast_target_attention_gb300 import workloads as W
from _helpers import MAX_ABS, MEAN_ABS, to_device

pytestmark = pytest.mark.gpu


def _call(fn, d, wl, out):
    n_cand, H, Lq, D = d["q"].shape
    rc = fn(d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(), d["user_offsets"].data_ptr(),
            d["cand_to_user"].data_ptr(), n_cand, wl.n_user, H, Lq, D, ctypes.c_float(wl.scale),
            out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return rc


@pytest.mark.parametrize("name", ["ratio_1024x15", "odd_groups_2048x16"])
def test_noalloc_matches_attn_fwd_on_two_calls_in_a_row(gpu_lib, name):
    lib = _lib.lib()
    wl = W.generate(W.CONFIGS[name])
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


def test_noalloc_rejects_a_call_that_needs_more_scratch(gpu_lib):
    """Many heads times many query tiles overflow the fixed array: refused, nothing run."""
    lib = _lib.lib()
    n_cand, n_user, H, Lq, D = 1 << 20, 1 << 20, 64, 128, 128
    A = 1 << 20
    # fake, never dereferenced addresses; out placed past the end of q
    rc = lib.ikbo_attn_fwd_noalloc(A, 2 * A, 3 * A, 4 * A, 5 * A, n_cand, n_user, H, Lq, D,
                                   ctypes.c_float(0.1), 1 << 44, None)
    assert rc == _lib.IKBO_ERR_SCRATCH
