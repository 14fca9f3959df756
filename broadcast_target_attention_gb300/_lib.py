"""ctypes declarations of the C ABI (include/ikbo.h).  Marshalling only."""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

_lock = threading.Lock()
_lib = None

STATUS = {
    0: "IKBO_OK", -1: "IKBO_ERR_NULL", -2: "IKBO_ERR_SHAPE", -3: "IKBO_ERR_ALIGN",
    -4: "IKBO_ERR_SCALE", -5: "IKBO_ERR_CUDA", -6: "IKBO_ERR_INDEX", -7: "IKBO_ERR_OFFSETS",
    -8: "IKBO_ERR_TIMEOUT", -9: "IKBO_ERR_ALIAS", -10: "IKBO_ERR_DEVICE", -11: "IKBO_ERR_BUDGET",
    -12: "IKBO_ERR_SCRATCH",
}
globals().update({name: code for code, name in STATUS.items()})

# name -> (restype, argtypes)
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_F = ctypes.c_float
SIGNATURES = {
    "ikbo_attn_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I32, _F, _P, _P]),
    "ikbo_broadcast_attn_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I32, _F,
                                                _P, ctypes.c_size_t, _P]),
    "ikbo_attn_fwd_host": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I32, _F, _P, _P]),
    "ikbo_get_device_error": (ctypes.c_int, [_P]),
    "ikbo_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "ikbo_version": (ctypes.c_int, []),
    "ikbo_shutdown": (ctypes.c_int, []),
    "ikbo_set_timing": (ctypes.c_int, [ctypes.c_int]),
    "ikbo_get_timing": (ctypes.c_int, [ctypes.POINTER(_F), ctypes.POINTER(_F)]),
    "ikbo_set_debug": (ctypes.c_int, [ctypes.c_int, ctypes.c_uint64]),
    "ikbo_set_kernel": (ctypes.c_int, [ctypes.c_int]),
    "ikbo_set_trace": (ctypes.c_int, [_P]),
    "ikbo_pool_usage": (ctypes.c_int, [ctypes.c_int, _P, _P]),
    "ikbo_launches_per_call": (ctypes.c_int, [_I64, _I64]),
    "ikbo_selected_kernel": (ctypes.c_int, [_I64, _I64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, _I64]),
    "ikbo_fused_attn_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _I32,
                                            _I32, _F, _P, _P, _P]),
    "ikbo_ml_attn_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _I32, _I32,
                                         _F, _P, _P]),
    "ikbo_ml_lce_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _I32,
                                        _I32, _I32, _I32, _P, _P]),
    "ikbo_lce_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I32, _I32, _P, _P]),
    "ikbo_attn_fwd_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _I64, _I64, _I32, _I32, _I32, _F,
                                              _P, _P]),
}


def lib():
    """The loaded library; raises if it has not been built (no fallback exists)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(_build.LIB):
                raise RuntimeError(
                    f"IKBO CUDA library missing ({_build.LIB}); build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'`")
            handle = ctypes.CDLL(_build.LIB)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(handle, name)
                fn.restype = res
                fn.argtypes = args
            _lib = handle
    return _lib
