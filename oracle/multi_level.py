"""CPU fp64 oracle for the multi-level broadcast -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may
import this module.  It shares no code with the CUDA path.

The hierarchy ("In-Kernel Broadcast Optimization: Co-Designing Kernels for
RecSys Inference", §5, conclusion and future directions): some recommendation
settings are deeper than user -> candidate, e.g. user -> ads vendor -> ads
item, where a user sees several vendors and each vendor offers several items.
Two broadcast relations are nested, with ratios that are independent of each
other and uneven.  The pages state that IKBO handles this structure but define
no operation on it, so the oracle takes the plainest reading for each of the
two IKBO primitives:

* target attention (§3): an item is a candidate.  Its Lq query tokens attend
  to the user sequence of the user its vendor belongs to, reached by walking
  the two maps: v = item_to_vendor[i], then u = vendor_to_user[v].
* linear compression (§2): an item's K input embeddings are its user's block,
  its vendor's block and its own block, concatenated along K, so
  out[i] = [W_user | W_vendor | W_item] @ [X_user[u]; X_vendor[v]; X_item[i]].
  Evaluated in that broadcast form, literally (both copies are made).

Every map value must lie in range (item_to_vendor in [0, n_vendor) and
vendor_to_user in [0, n_user)); an out-of-range value raises ValueError.
"""
from __future__ import annotations

import numpy as np


def _f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def walk(item_to_vendor, vendor_to_user, n_user: int) -> np.ndarray:
    """The user of every item: its vendor's user.  int64 [n_item]."""
    i2v = np.asarray(item_to_vendor, dtype=np.int64)
    v2u = np.asarray(vendor_to_user, dtype=np.int64)
    if np.any(i2v < 0) or np.any(i2v >= v2u.shape[0]):
        raise ValueError("multi-level oracle: item_to_vendor out of range")
    if np.any(v2u < 0) or np.any(v2u >= n_user):
        raise ValueError("multi-level oracle: vendor_to_user out of range")
    users = np.empty(i2v.shape[0], dtype=np.int64)
    for i, v in enumerate(i2v.tolist()):
        users[i] = v2u[v]
    return users


def attention(q, k, v, user_offsets, item_to_vendor, vendor_to_user, scale: float,
              items=None) -> np.ndarray:
    """fp64 target attention of every item (or the selected ``items``) over its user's
    sequence: the two maps walked per item, then the two-level target attention (the C
    oracle) with that user.  q: uint16 [n_item, H, Lq, D]; k, v: uint16 [T, H, D]."""
    from . import attention as target_attention
    n_user = int(np.asarray(user_offsets).shape[0]) - 1
    users = walk(item_to_vendor, vendor_to_user, n_user).astype(np.int32)
    return target_attention(q, k, v, user_offsets, users, scale, items)


def lce(W_user, W_vendor, W_item, X_user, X_vendor, X_item, item_to_vendor, vendor_to_user,
        items=None) -> np.ndarray:
    """out[i] = [W_user | W_vendor | W_item] @ [X_user[u(i)]; X_vendor[v(i)]; X_item[i]] in
    float64, for every item (or the selected ``items``).  Any K block may be empty."""
    n_user = X_user.shape[0]
    users = walk(item_to_vendor, vendor_to_user, n_user)
    i2v = np.asarray(item_to_vendor, dtype=np.int64)
    W = np.concatenate([_f64(W_user), _f64(W_vendor), _f64(W_item)], axis=1)
    n_item = X_item.shape[0]
    sel = np.arange(n_item) if items is None else np.asarray(items, dtype=np.int64)
    M, N = W.shape[0], X_item.shape[2]
    out = np.empty((len(sel), M, N), dtype=np.float64)
    for j, i in enumerate(sel.tolist()):
        # the broadcast at both levels: this item's own copies of its user's and vendor's blocks
        X = np.concatenate([_f64(X_user[users[i]]), _f64(X_vendor[i2v[i]]), _f64(X_item[i])], axis=0)
        out[j] = W @ X
    return out
