"""The C ABI without a GPU: the library loads, exports what include/ikbo.h
declares, and rejects bad host-visible arguments before touching CUDA."""
import os
import re

import pytest

import broadcast_target_attention_gb300 as ikbo
from broadcast_target_attention_gb300 import _lib
from broadcast_target_attention_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    B.build()
    return _lib.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "ikbo.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(ikbo_[a-z_]+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("ikbo_attn_fwd", "ikbo_broadcast_attn_fwd", "ikbo_attn_fwd_host",
                     "ikbo_get_device_error", "ikbo_strerror", "ikbo_version"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, f"{name} has no ctypes signature"


def test_version_and_strerror(lib):
    assert lib.ikbo_version() >= 10000
    for code in _lib.STATUS:
        assert lib.ikbo_strerror(code)
    assert lib.ikbo_strerror(12345) == b"unknown status"


def test_launches_per_call(lib):
    assert lib.ikbo_launches_per_call(0, 5) == 0
    assert lib.ikbo_launches_per_call(1024, 15) == 1         # planning fused into the kernel
    assert lib.ikbo_launches_per_call(20480, 1024) == 1
    assert lib.ikbo_launches_per_call(20481, 15) == 2        # separate planning launch
    assert lib.ikbo_launches_per_call(1024, 1025) == 2
    assert lib.ikbo_launches_per_call(-1, 2) == _lib.IKBO_ERR_SHAPE
    prev = lib.ikbo_set_kernel(1)
    try:
        assert lib.ikbo_launches_per_call(1024, 15) == 2     # SIMT kernel: always planned apart
    finally:
        lib.ikbo_set_kernel(prev)


A = 1 << 20   # a fake, 16-byte aligned "device" address; never dereferenced


def call(lib, q=A, k=2 * A, v=3 * A, off=4 * A, c2u=5 * A, n_cand=8, n_user=2, H=2, Lq=1, D=64,
         scale=0.125, out=6 * A):
    return lib.ikbo_attn_fwd(q, k, v, off, c2u, n_cand, n_user, H, Lq, D, scale, out, None)


def test_host_detectable_errors_return_before_any_cuda_call(lib):
    assert call(lib, D=96) == _lib.IKBO_ERR_SHAPE
    assert call(lib, Lq=0) == _lib.IKBO_ERR_SHAPE
    assert call(lib, Lq=129) == _lib.IKBO_ERR_SHAPE
    assert call(lib, H=0) == _lib.IKBO_ERR_SHAPE
    assert call(lib, n_cand=-1) == _lib.IKBO_ERR_SHAPE
    assert call(lib, n_user=-1) == _lib.IKBO_ERR_SHAPE
    assert call(lib, scale=float("inf")) == _lib.IKBO_ERR_SCALE
    assert call(lib, scale=float("nan")) == _lib.IKBO_ERR_SCALE
    assert call(lib, q=None) == _lib.IKBO_ERR_NULL
    assert call(lib, out=None) == _lib.IKBO_ERR_NULL
    assert call(lib, c2u=None) == _lib.IKBO_ERR_NULL
    assert call(lib, k=2 * A + 8) == _lib.IKBO_ERR_ALIGN
    assert call(lib, off=4 * A + 2) == _lib.IKBO_ERR_ALIGN
    assert call(lib, out=A + 64) == _lib.IKBO_ERR_ALIAS      # overlaps q
    assert call(lib, n_user=0) == _lib.IKBO_ERR_INDEX         # nothing to map candidates to
    assert call(lib, n_cand=0, q=None, out=None) == _lib.IKBO_OK   # empty batch: no-op


def test_broadcast_and_host_paths_check_arguments_too(lib):
    rc = lib.ikbo_broadcast_attn_fwd(A, 2 * A, 3 * A, 4 * A, 5 * A, 8, 2, 2, 1, 80, 0.1, 6 * A,
                                     1 << 30, None)
    assert rc == _lib.IKBO_ERR_SHAPE
    rc = lib.ikbo_attn_fwd_host(A, 2 * A, 3 * A, 4 * A, 5 * A, 8, 2, 2, 1, 64, float("inf"), 6 * A,
                                None)
    assert rc == _lib.IKBO_ERR_SCALE


def test_python_binding_raises_on_bad_status(lib):
    with pytest.raises(ikbo.IkboError) as e:
        ikbo._check(_lib.IKBO_ERR_SHAPE, "x")
    assert "IKBO_ERR_SHAPE" in str(e.value)


def test_selected_kernel(lib):
    """Automatic choice: two query tiles per item when the users have on average at least
    two query tiles each, the batch makes at least 600 two-tile items (200 for target
    attention alone at D = 128 with at most 256 users) and the inputs fit the in-kernel
    planning limits; the key-interleaved kernel (4) only when chosen; a fused call on the
    one- or two-tile kernel."""
    sel = lib.ikbo_selected_kernel
    assert sel(1024, 15, 4, 1, 128, -1) == 2      # 1024 candidates / 15 users, Lq 1: < 1 tile per user
    assert sel(8, 2, 2, 1, 64, -1) == 2
    assert sel(2048, 16, 8, 4, 128, -1) == 3      # 4 tiles per user, 256 items, D 128
    assert sel(2048, 16, 8, 4, 64, -1) == 2       # the same at D 64
    assert sel(2048, 16, 8, 4, 128, 34855) == 2   # the same, fused with self-attention
    assert sel(1600, 16, 8, 4, 128, -1) == 3      # exactly 200 items
    assert sel(1000, 16, 16, 4, 128, -1) == 2     # 256 items, fewer than two tiles per user
    assert sel(8192, 256, 1, 8, 128, -1) == 3     # 256 items of 256 users
    assert sel(8224, 257, 1, 8, 128, -1) == 2     # 257 items of 257 users
    assert sel(6336, 99, 1, 8, 128, -1) == 2      # 198 items
    assert sel(4096, 4, 8, 8, 128, -1) == 3       # 64 tiles per user, 1024 items
    assert sel(4096, 4, 8, 8, 64, 20000) == 3     # ... fused too
    assert sel(16384, 64, 16, 1, 64, -1) == 3     # exactly two tiles per user, 1024 items
    assert sel(16383, 64, 16, 1, 64, -1) == 2
    assert sel(16384, 64, 16, 4, 128, -1) == 3
    assert sel(16384, 64, 2, 1, 128, -1) == 2     # 128 items
    assert sel(20481, 4, 8, 8, 128, -1) == 2      # beyond the in-kernel planning limits
    assert sel(4096, 1025, 8, 1, 128, -1) == 2
    assert sel(-1, 2, 1, 1, 64, -1) == _lib.IKBO_ERR_SHAPE
    assert sel(8, 2, 0, 1, 64, -1) == _lib.IKBO_ERR_SHAPE
    assert sel(8, 2, 1, 0, 64, -1) == _lib.IKBO_ERR_SHAPE
    assert sel(8, 2, 1, 129, 64, -1) == _lib.IKBO_ERR_SHAPE
    assert sel(8, 2, 1, 1, 96, -1) == _lib.IKBO_ERR_SHAPE
    for which, expect, fused in ((1, 1, 2), (2, 2, 2), (3, 3, 3), (4, 4, 2), (7, 2, 2)):
        prev = lib.ikbo_set_kernel(which)
        try:
            assert sel(1024, 15, 4, 1, 128, -1) == expect
            assert sel(1024, 15, 4, 1, 128, 9000) == fused
            assert sel(20481, 4, 8, 8, 128, -1) == (1 if which == 1 else 2)   # two tiles: in-kernel planning only
            assert lib.ikbo_launches_per_call(1024, 15) == (2 if which == 1 else 1)
        finally:
            lib.ikbo_set_kernel(prev)


def test_shutdown_without_any_device_set_up(lib):
    """Nothing set up in this process: no CUDA call, and OK (twice)."""
    assert lib.ikbo_shutdown() == 0
    assert lib.ikbo_shutdown() == 0
