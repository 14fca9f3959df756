"""CPU fp64 oracle for IKBO target attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg
(and its ``--impl reference`` arm) may import this package.  The product path
(the CUDA library and its binding) never calls it and shares no code with it.

``ikbo_oracle.c`` holds the arithmetic; this module compiles it with gcc
(OpenMP, no other dependency) and calls it through ctypes.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ikbo_oracle.c")
_LIB = os.path.join(_HERE, "libikbo_oracle.so")
_lock = threading.Lock()
_lib = None

ERRORS = {0: "ok", -1: "bad argument", -2: "cand_to_user out of range",
          -3: "user_offsets not a valid jagged index", -4: "out of memory"}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/libikbo_oracle.so`` (skipped when fresh)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall", "-Wextra",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            i32 = ctypes.c_int32
            lib.ikbo_oracle_fwd.argtypes = [p, p, p, p, p, i64, i64, i32, i32, i32,
                                            ctypes.c_double, p, i64, p]
            lib.ikbo_oracle_fwd.restype = ctypes.c_int
            lib.ikbo_oracle_weights.argtypes = [p, p, p, p, i64, i64, i32, i32, i32,
                                                ctypes.c_double, i64, i32, i32, p]
            lib.ikbo_oracle_weights.restype = ctypes.c_int
            lib.ikbo_oracle_self_fwd.argtypes = [p, p, p, p, i64, i32, i32, ctypes.c_double, p, i64,
                                                 p]
            lib.ikbo_oracle_self_fwd.restype = ctypes.c_int
            lib.ikbo_oracle_num_threads.argtypes = []
            lib.ikbo_oracle_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _prep(q, k, v, user_offsets, cand_to_user):
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16) if v is not None else None
    off = np.ascontiguousarray(user_offsets, dtype=np.int32)
    c2u = np.ascontiguousarray(cand_to_user, dtype=np.int32)
    return q, k, v, off, c2u


def attention(q, k, v, user_offsets, cand_to_user, scale: float, cands=None) -> np.ndarray:
    """fp64 target attention for the selected candidates (all when ``cands`` is None).

    q: uint16 bf16 bits [n_cand, H, Lq, D]; k, v: uint16 [T, H, D];
    returns float64 [n_sel, H, Lq, D].
    """
    q, k, v, off, c2u = _prep(q, k, v, user_offsets, cand_to_user)
    n_cand, H, Lq, D = q.shape
    n_user = off.shape[0] - 1
    if cands is None:
        sel = None
        n_sel = n_cand
    else:
        sel = np.ascontiguousarray(cands, dtype=np.int64)
        n_sel = sel.shape[0]
    out = np.zeros((n_sel, H, Lq, D), dtype=np.float64)
    rc = _load().ikbo_oracle_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(off), _ptr(c2u), n_cand, n_user,
                                 H, Lq, D, float(scale), _ptr(sel) if sel is not None else None,
                                 n_sel, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle: {ERRORS.get(rc, rc)}")
    return out


def attention_wl(wl, cands=None) -> np.ndarray:
    """``attention`` on a ``workloads.Workload``."""
    return attention(wl.q, wl.k, wl.v, wl.user_offsets, wl.cand_to_user, wl.scale, cands)


def weights(q, k, user_offsets, cand_to_user, scale: float, c: int, h: int, t: int) -> np.ndarray:
    """The attention weights of one query row (candidate c, head h, token t)."""
    q, k, _, off, c2u = _prep(q, k, None, user_offsets, cand_to_user)
    n_cand, H, Lq, D = q.shape
    n_user = off.shape[0] - 1
    u = int(c2u[c])
    L = int(off[u + 1]) - int(off[u])
    probs = np.zeros(max(L, 1), dtype=np.float64)
    rc = _load().ikbo_oracle_weights(_ptr(q), _ptr(k), _ptr(off), _ptr(c2u), n_cand, n_user, H, Lq,
                                     D, float(scale), int(c), int(h), int(t), _ptr(probs))
    if rc != 0:
        raise ValueError(f"oracle: {ERRORS.get(rc, rc)}")
    return probs[:L]


def self_attention(q_user, k, v, user_offsets, scale: float, rows=None) -> np.ndarray:
    """fp64 self-attention of the user sequence over itself (full, no causal mask), for the
    selected sequence rows (all when ``rows`` is None).

    q_user, k, v: uint16 bf16 bits [T, H, D]; returns float64 [n_sel, H, D].
    """
    qu = np.ascontiguousarray(q_user, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    off = np.ascontiguousarray(user_offsets, dtype=np.int32)
    T, H, D = qu.shape
    if k.shape != qu.shape or v.shape != qu.shape:
        raise ValueError("oracle: q_user, k and v must share [T, H, D]")
    n_user = off.shape[0] - 1
    if rows is None:
        sel = None
        n_sel = T
    else:
        sel = np.ascontiguousarray(rows, dtype=np.int64)
        n_sel = sel.shape[0]
    out = np.zeros((n_sel, H, D), dtype=np.float64)
    rc = _load().ikbo_oracle_self_fwd(_ptr(qu), _ptr(k), _ptr(v), _ptr(off), n_user, H, D,
                                      float(scale), _ptr(sel) if sel is not None else None, n_sel,
                                      _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle: {ERRORS.get(rc, rc)}")
    return out


def lce(W_user, W_cand, X_user, X_cand, cand_to_user, cands=None) -> np.ndarray:
    """fp64 IKBO linear compression (see ``oracle/linear_compression.py``)."""
    from . import linear_compression
    return linear_compression.lce(W_user, W_cand, X_user, X_cand, cand_to_user, cands)


def ml_attention(q, k, v, user_offsets, item_to_vendor, vendor_to_user, scale: float,
                 items=None) -> np.ndarray:
    """fp64 target attention over a user -> vendor -> item hierarchy (see
    ``oracle/multi_level.py``)."""
    from . import multi_level
    return multi_level.attention(q, k, v, user_offsets, item_to_vendor, vendor_to_user, scale, items)


def ml_lce(W_user, W_vendor, W_item, X_user, X_vendor, X_item, item_to_vendor, vendor_to_user,
           items=None) -> np.ndarray:
    """fp64 linear compression over a user -> vendor -> item hierarchy (see
    ``oracle/multi_level.py``)."""
    from . import multi_level
    return multi_level.lce(W_user, W_vendor, W_item, X_user, X_vendor, X_item, item_to_vendor,
                           vendor_to_user, items)


def num_threads() -> int:
    """OpenMP threads the oracle runs on (OMP_NUM_THREADS, else all cores)."""
    return int(_load().ikbo_oracle_num_threads())
