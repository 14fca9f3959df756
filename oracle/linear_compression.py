"""CPU fp64 oracle for IKBO linear compression -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the bench's CPU-baseline leg may
import this module.  It shares no code with the CUDA path.

Definition followed ("In-Kernel Broadcast Optimization: Co-Designing Kernels for
RecSys Inference", §2 and §2.1 with Fig. 2): linear compression of embeddings
(LCE) projects each candidate's input embeddings X[b] (K x N) with a learned
W (M x K): out[b] = W @ X[b], an (M, K) @ (B, K, N) -> (B, M, N) batched
matrix product.  The K embeddings of a candidate are its user's block
followed by its own block, concatenated along K, so for candidate b of user
u = cand_to_user[b]:

    out[b] = W @ [ X_user[u] ; X_cand[b] ]          W = [ W_user | W_cand ]

This module evaluates that broadcast form literally (it builds the
concatenated X[b] for every selected candidate, copying the user block) in
float64 from the exact bf16 input values; numpy's matmul is the product.
IKBO computes the same result as W_user @ X_user[u] + W_cand @ X_cand[b]
(§2.1: the broadcast pushed past the matrix product), equal up to rounding.

Layouts (bf16 as raw uint16 bits): W_user [M, K_user], W_cand [M, K_cand],
X_user [n_user, K_user, N], X_cand [n_cand, K_cand, N]; result float64
[n_sel, M, N] for the selected candidates (all when ``cands`` is None).
"""
from __future__ import annotations

import numpy as np


def _f64(bits: np.ndarray) -> np.ndarray:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def lce(W_user, W_cand, X_user, X_cand, cand_to_user, cands=None) -> np.ndarray:
    """out[b] = [W_user | W_cand] @ [X_user[u(b)] ; X_cand[b]] in float64."""
    Wu, Wc = _f64(W_user), _f64(W_cand)
    c2u = np.asarray(cand_to_user, dtype=np.int64)
    n_cand = X_cand.shape[0]
    n_user = X_user.shape[0]
    if np.any(c2u < 0) or np.any(c2u >= n_user):
        raise ValueError("lce oracle: cand_to_user out of range")
    W = np.concatenate([Wu, Wc], axis=1)                       # [M, K_user + K_cand]
    sel = np.arange(n_cand) if cands is None else np.asarray(cands, dtype=np.int64)
    M, N = W.shape[0], X_cand.shape[2]
    out = np.empty((len(sel), M, N), dtype=np.float64)
    for i, b in enumerate(sel.tolist()):
        # the broadcast: this candidate's own copy of its user's block, then its block
        X = np.concatenate([_f64(X_user[c2u[b]]), _f64(X_cand[b])], axis=0)
        out[i] = W @ X
    return out
