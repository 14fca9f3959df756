"""IKBO target attention on GB300 (sm_103a): Python binding of the C ABI.

Every function here only checks and marshals arguments (tensor pointers,
sizes, the current CUDA stream) and calls ``libikbo.so``; all arithmetic runs
in the library's CUDA kernels.  There is no CPU or PyTorch fallback: if the
library is missing the call raises.

Layouts (see include/ikbo.h): q/out bf16 [n_cand, H, Lq, D]; k/v bf16
[T, H, D] packed by user; user_offsets int32 [n_user+1]; cand_to_user int32
[n_cand].  Besides the target attention: the fused self + target call, the
user -> vendor -> item hierarchy (attention and linear compression), IKBO
linear compression, the explicit-broadcast comparison path, the host-buffer
and allocation-free entry points.
"""
from __future__ import annotations

import ctypes
from typing import Optional, Tuple

from . import _lib
from ._lib import STATUS

__all__ = ["attn_fwd", "fused_attn_fwd", "ml_attn_fwd", "lce_fwd", "ml_lce_fwd", "broadcast_attn_fwd",
           "attn_fwd_host", "attn_fwd_noalloc", "get_device_error", "set_timing", "get_timing",
           "set_kernel", "selected_kernel", "set_debug", "set_trace", "launches_per_call", "version",
           "shutdown", "pool_usage", "load", "IkboError", "STATUS"]


class IkboError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        msg = _lib.lib().ikbo_strerror(status).decode()
        super().__init__(f"{STATUS.get(status, status)}: {msg}" + (f" ({what})" if what else ""))


def load():
    """Load the CUDA library (raises if it was not built)."""
    return _lib.lib()


def _check(rc: int, what: str = "") -> None:
    if rc != 0:
        raise IkboError(rc, what)


def _ptr(t) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _shape(q, k):
    if q.dim() != 4 or k.dim() != 3:
        raise ValueError("q must be [n_cand, H, Lq, D] and k/v [T, H, D]")
    n_cand, H, Lq, D = q.shape
    if k.shape[1] != H or k.shape[2] != D:
        raise ValueError(f"k shape {tuple(k.shape)} does not match q heads/dim ({H}, {D})")
    return int(n_cand), int(H), int(Lq), int(D)


def _validate(q, k, v, user_offsets, cand_to_user, device: bool):
    import torch
    for name, t, dt in (("q", q, torch.bfloat16), ("k", k, torch.bfloat16), ("v", v, torch.bfloat16),
                        ("user_offsets", user_offsets, torch.int32),
                        ("cand_to_user", cand_to_user, torch.int32)):
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
        if device and not t.is_cuda:
            raise ValueError(f"{name} must be a CUDA tensor")
        if not device and t.is_cuda:
            raise ValueError(f"{name} must be a host tensor")
    if v.shape != k.shape:
        raise ValueError("k and v must have the same shape")


def attn_fwd(q, k, v, user_offsets, cand_to_user, scale: Optional[float] = None, out=None,
             stream=None):
    """IKBO target attention on device tensors; returns ``out`` (bf16, like q).

    Asynchronous on ``stream`` (default: torch's current stream).  Index
    errors found on the GPU are reported by :func:`get_device_error`.
    """
    import torch
    _validate(q, k, v, user_offsets, cand_to_user, device=True)
    n_cand, H, Lq, D = _shape(q, k)
    n_user = int(user_offsets.shape[0]) - 1
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    rc = _lib.lib().ikbo_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(user_offsets), _ptr(cand_to_user),
                                  n_cand, n_user, H, Lq, D, float(scale), _ptr(out),
                                  _stream_handle(stream))
    _check(rc, "ikbo_attn_fwd")
    return out


def ml_attn_fwd(q, k, v, user_offsets, item_to_vendor, vendor_to_user,
                scale: Optional[float] = None, out=None, stream=None):
    """Target attention over a user -> vendor -> item hierarchy (device tensors): item i
    attends to the sequence of user ``vendor_to_user[item_to_vendor[i]]``; returns ``out``.
    See ``ikbo_ml_attn_fwd`` in include/ikbo.h."""
    import torch
    _validate(q, k, v, user_offsets, item_to_vendor, device=True)
    if (vendor_to_user.dtype != torch.int32 or not vendor_to_user.is_contiguous()
            or not vendor_to_user.is_cuda):
        raise ValueError("vendor_to_user must be a contiguous int32 CUDA tensor")
    n_item, H, Lq, D = _shape(q, k)
    n_user = int(user_offsets.shape[0]) - 1
    n_vendor = int(vendor_to_user.shape[0])
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    rc = _lib.lib().ikbo_ml_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(user_offsets),
                                     _ptr(item_to_vendor), _ptr(vendor_to_user), n_item, n_vendor,
                                     n_user, H, Lq, D, float(scale), _ptr(out),
                                     _stream_handle(stream))
    _check(rc, "ikbo_ml_attn_fwd")
    return out


def fused_attn_fwd(q, q_user, k, v, user_offsets, cand_to_user, scale: Optional[float] = None,
                   out=None, out_user=None, stream=None):
    """Target attention of the candidates and self-attention of the user sequence in one
    launch (device tensors); returns ``(out, out_user)``.

    ``q_user`` is bf16 ``[T, H, D]`` like ``k``; ``q`` may have zero candidates.  See
    ``ikbo_fused_attn_fwd`` in include/ikbo.h.
    """
    import torch
    _validate(q, k, v, user_offsets, cand_to_user, device=True)
    if q_user.dtype != torch.bfloat16 or not q_user.is_contiguous() or not q_user.is_cuda:
        raise ValueError("q_user must be a contiguous bf16 CUDA tensor")
    if q_user.shape != k.shape:
        raise ValueError("q_user must have the shape of k, [T, H, D]")
    T, H, D = (int(x) for x in k.shape)
    n_cand = int(q.shape[0])
    Lq = int(q.shape[2]) if q.dim() == 4 else 1
    if n_cand and (q.dim() != 4 or int(q.shape[1]) != H or int(q.shape[3]) != D):
        raise ValueError("q must be [n_cand, H, Lq, D] with the H and D of k")
    n_user = int(user_offsets.shape[0]) - 1
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    if out_user is None:
        out_user = torch.empty_like(q_user)
    p = lambda t: _ptr(t) if t.numel() else None
    rc = _lib.lib().ikbo_fused_attn_fwd(p(q), p(q_user), p(k), p(v), _ptr(user_offsets),
                                        p(cand_to_user), n_cand, n_user, T, H, Lq, D, float(scale),
                                        p(out), p(out_user), _stream_handle(stream))
    _check(rc, "ikbo_fused_attn_fwd")
    return out, out_user


def lce_fwd(W_user, W_cand, X_user, X_cand, cand_to_user, out=None, stream=None):
    """IKBO linear compression on device tensors (see ``ikbo_lce_fwd`` in include/ikbo.h):
    ``out[b] = W_user @ X_user[cand_to_user[b]] + W_cand @ X_cand[b]``; returns ``out``."""
    import torch
    for name, t in (("W_cand", W_cand), ("X_cand", X_cand), ("W_user", W_user), ("X_user", X_user)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if cand_to_user.dtype != torch.int32 or not cand_to_user.is_contiguous() or not cand_to_user.is_cuda:
        raise ValueError("cand_to_user must be a contiguous int32 CUDA tensor")
    n_cand, K_cand, N = (int(x) for x in X_cand.shape)
    n_user, K_user = int(X_user.shape[0]), int(X_user.shape[1])
    M = int(W_cand.shape[0])
    if W_cand.shape != (M, K_cand) or W_user.shape != (M, K_user) or X_user.shape[2] != N:
        raise ValueError("shapes: W_user [M, K_user], W_cand [M, K_cand], X_user [n_user, K_user, N], "
                         "X_cand [n_cand, K_cand, N]")
    if out is None:
        out = torch.empty((n_cand, M, N), dtype=torch.bfloat16, device=X_cand.device)
    p = lambda t: _ptr(t) if t.numel() else None
    rc = _lib.lib().ikbo_lce_fwd(p(W_user), p(W_cand), p(X_user), p(X_cand), p(cand_to_user), n_cand,
                                 n_user, M, K_user, K_cand, N, p(out), _stream_handle(stream))
    _check(rc, "ikbo_lce_fwd")
    return out


def ml_lce_fwd(W_user, W_vendor, W_item, X_user, X_vendor, X_item, item_to_vendor,
               vendor_to_user, out=None, stream=None):
    """Linear compression over a user -> vendor -> item hierarchy on device tensors (see
    ``ikbo_ml_lce_fwd`` in include/ikbo.h): ``out[i] = W_user @ X_user[u] + W_vendor @
    X_vendor[v] + W_item @ X_item[i]`` with ``v = item_to_vendor[i]``, ``u =
    vendor_to_user[v]``; returns ``out``.  A block with K = 0 is left out."""
    import torch
    for name, t in (("W_user", W_user), ("W_vendor", W_vendor), ("W_item", W_item),
                    ("X_user", X_user), ("X_vendor", X_vendor), ("X_item", X_item)):
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    for name, t in (("item_to_vendor", item_to_vendor), ("vendor_to_user", vendor_to_user)):
        if t.dtype != torch.int32 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous int32 CUDA tensor")
    n_item, K_item, N = (int(x) for x in X_item.shape)
    n_vendor, K_vendor = int(X_vendor.shape[0]), int(X_vendor.shape[1])
    n_user, K_user = int(X_user.shape[0]), int(X_user.shape[1])
    M = int(W_item.shape[0])
    if (W_item.shape != (M, K_item) or W_vendor.shape != (M, K_vendor) or W_user.shape != (M, K_user)
            or X_vendor.shape[2] != N or X_user.shape[2] != N
            or tuple(item_to_vendor.shape) != (n_item,) or tuple(vendor_to_user.shape) != (n_vendor,)):
        raise ValueError("shapes: W_* [M, K_*], X_user [n_user, K_user, N], X_vendor [n_vendor, "
                         "K_vendor, N], X_item [n_item, K_item, N], item_to_vendor [n_item], "
                         "vendor_to_user [n_vendor]")
    if out is None:
        out = torch.empty((n_item, M, N), dtype=torch.bfloat16, device=X_item.device)
    p = lambda t: _ptr(t) if t.numel() else None
    rc = _lib.lib().ikbo_ml_lce_fwd(p(W_user), p(W_vendor), p(W_item), p(X_user), p(X_vendor),
                                    p(X_item), p(item_to_vendor), p(vendor_to_user), n_item,
                                    n_vendor, n_user, M, K_user, K_vendor, K_item, N, p(out),
                                    _stream_handle(stream))
    _check(rc, "ikbo_ml_lce_fwd")
    return out


def broadcast_attn_fwd(q, k, v, user_offsets, cand_to_user, scale: Optional[float] = None,
                       out=None, mem_budget_bytes: int = 16 << 30, stream=None):
    """The explicit-broadcast comparison path (copies K/V per candidate first)."""
    import torch
    _validate(q, k, v, user_offsets, cand_to_user, device=True)
    n_cand, H, Lq, D = _shape(q, k)
    n_user = int(user_offsets.shape[0]) - 1
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    rc = _lib.lib().ikbo_broadcast_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(user_offsets),
                                            _ptr(cand_to_user), n_cand, n_user, H, Lq, D,
                                            float(scale), _ptr(out), int(mem_budget_bytes),
                                            _stream_handle(stream))
    _check(rc, "ikbo_broadcast_attn_fwd")
    return out


def attn_fwd_host(q, k, v, user_offsets, cand_to_user, scale: Optional[float] = None, out=None,
                  stream=None):
    """IKBO target attention on HOST tensors (pinned recommended); synchronous.

    The library copies the inputs to the GPU, runs, and copies ``out`` back.
    """
    import torch
    _validate(q, k, v, user_offsets, cand_to_user, device=False)
    n_cand, H, Lq, D = _shape(q, k)
    n_user = int(user_offsets.shape[0]) - 1
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    rc = _lib.lib().ikbo_attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(user_offsets),
                                       _ptr(cand_to_user), n_cand, n_user, H, Lq, D, float(scale),
                                       _ptr(out), _stream_handle(stream))
    _check(rc, "ikbo_attn_fwd_host")
    return out


def attn_fwd_noalloc(q, k, v, user_offsets, cand_to_user, scale: Optional[float] = None, out=None,
                     stream=None):
    """attn_fwd whose scratch comes from the library's fixed device array, not
    from an allocation (for callers whose memory manager forbids the library
    to allocate); see ikbo_attn_fwd_noalloc in include/ikbo.h.  ``out`` must
    be passed in by such callers to avoid the allocation of a new tensor."""
    import torch
    _validate(q, k, v, user_offsets, cand_to_user, device=True)
    n_cand, H, Lq, D = _shape(q, k)
    n_user = int(user_offsets.shape[0]) - 1
    if scale is None:
        scale = D ** -0.5
    if out is None:
        out = torch.empty_like(q)
    rc = _lib.lib().ikbo_attn_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(user_offsets),
                                          _ptr(cand_to_user), n_cand, n_user, H, Lq, D,
                                          float(scale), _ptr(out), _stream_handle(stream))
    _check(rc, "ikbo_attn_fwd_noalloc")
    return out


def pool_usage(reset: bool = False) -> Tuple[int, int]:
    """(bytes held now, most bytes held at once since the last reset) of the library's own
    stream-ordered pool on the current device; ``reset`` restarts the high-water mark
    (test hook, see ikbo_pool_usage in include/ikbo.h)."""
    now = ctypes.c_uint64()
    high = ctypes.c_uint64()
    _check(_lib.lib().ikbo_pool_usage(1 if reset else 0, ctypes.byref(now), ctypes.byref(high)),
           "ikbo_pool_usage")
    return now.value, high.value


def get_device_error(stream=None) -> int:
    """Synchronise the stream; return and clear the device error word (0 = none)."""
    return int(_lib.lib().ikbo_get_device_error(_stream_handle(stream)))


def set_timing(enable: bool) -> None:
    _check(_lib.lib().ikbo_set_timing(1 if enable else 0))


def get_timing() -> Tuple[float, float]:
    """(planning kernel ms, attention kernel ms) of the last timed call."""
    a = ctypes.c_float()
    b = ctypes.c_float()
    _check(_lib.lib().ikbo_get_timing(ctypes.byref(a), ctypes.byref(b)), "ikbo_get_timing")
    return a.value, b.value


# kernel choices of set_kernel / results of selected_kernel
KERNEL_AUTO, KERNEL_SIMT, KERNEL_TC, KERNEL_TC2, KERNEL_AB = 0, 1, 2, 3, 4
KERNEL_NAMES = {KERNEL_SIMT: "ikbo_attn_simt_kernel", KERNEL_TC: "ikbo_attn_tc_kernel",
                KERNEL_TC2: "ikbo_attn_pp_kernel", KERNEL_AB: "ikbo_attn_ab_kernel"}


def set_kernel(which: int) -> int:
    """0 = automatic (default), 1 = SIMT cross-check kernel, 2 = tcgen05 kernel with one
    query tile per work item, 3 = tcgen05 kernel with two query tiles of one user and head
    per work item, 4 = tcgen05 kernel with the key tiles of one query tile over two softmax
    warpgroups; returns the previous choice."""
    return int(_lib.lib().ikbo_set_kernel(int(which)))


def selected_kernel(n_cand: int, n_user: int, H: int, Lq: int, D: int, self_rows: int = -1) -> int:
    """The kernel (1 to 4) that attn_fwd (self_rows < 0) or fused_attn_fwd over self_rows
    sequence rows runs with these sizes and this thread's choice."""
    n = int(_lib.lib().ikbo_selected_kernel(int(n_cand), int(n_user), int(H), int(Lq), int(D),
                                            int(self_rows)))
    _check(min(n, 0), "selected_kernel")
    return n


def launches_per_call(n_cand: int, n_user: int) -> int:
    """Kernel launches one attn_fwd call makes for this batch size (host arithmetic only)."""
    n = int(_lib.lib().ikbo_launches_per_call(int(n_cand), int(n_user)))
    _check(min(n, 0), "launches_per_call")
    return n


def set_debug(flags: int = 0, timeout_ns: int = 0) -> None:
    """Test hook of the library (see ikbo_set_debug in include/ikbo.h)."""
    _check(_lib.lib().ikbo_set_debug(int(flags), int(timeout_ns)))


def set_trace(buffer) -> None:
    """Trace the tcgen05 kernel into ``buffer`` (a CUDA uint64/int64 tensor of
    at least SMs*4*16 entries), or stop tracing with None."""
    _check(_lib.lib().ikbo_set_trace(None if buffer is None else buffer.data_ptr()))


def version() -> int:
    return int(_lib.lib().ikbo_version())


def shutdown() -> None:
    """Release the library's per-device resources and trim the memory pools it used (see
    ``ikbo_shutdown`` in include/ikbo.h); the next call sets a device up again."""
    _check(_lib.lib().ikbo_shutdown(), "ikbo_shutdown")
