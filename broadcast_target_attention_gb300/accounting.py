"""Work and traffic accounting for IKBO target attention and linear compression
(host arithmetic only).

FLOPs count the two contractions (Q·Kᵀ and P·V), 2 FLOPs per multiply-add,
softmax excluded -- the convention of "In-Kernel Broadcast Optimization:
Co-Designing Kernels for RecSys Inference", Appendix 9 (roofline of standard
vs IKBO flash attention) and Appendix 2 (arithmetic intensity = FLOPs over
bytes moved to and from HBM).

Algorithmic bytes are what an ideal IKBO kernel must move: every user K/V row
read once, every query read once, every output written once, plus the index
tensors.  The explicit-broadcast comparison path additionally writes the
per-candidate K/V copy and reads it back.
"""
from __future__ import annotations

BF16 = 2


def flops(H: int, D: int, Lq: int, S: int) -> int:
    """4·H·D·Lq·S, with S = Σ_c L_{u(c)} keys visited over all candidates."""
    return 4 * H * D * Lq * S


def alg_bytes(H: int, D: int, Lq: int, T: int, n_cand: int, n_user: int) -> int:
    """K and V read once per user, q read and out written once, int32 indices."""
    kv = 2 * T * H * D * BF16
    q_out = 2 * n_cand * H * Lq * D * BF16
    idx = 4 * (n_cand + n_user + 1)
    return kv + q_out + idx


def broadcast_extra_bytes(H: int, D: int, S_tokens: int) -> int:
    """Extra traffic of the explicit broadcast: write the K/V copy, read it back."""
    return 2 * (2 * S_tokens * H * D * BF16)


def ai_per_user_head(r: int, Lq: int, L: int) -> float:
    """Arithmetic intensity (FLOP/B) of one user-head with r candidates.

    FLOPs 4·D·r·Lq·L over bytes 2·D·(2L + 2·r·Lq): K/V of the user read once,
    each candidate's queries read and outputs written once.  r = 1 is the
    standard (broadcast) kernel, whose K/V are re-read for every candidate.
    """
    return r * Lq * L / (L + r * Lq)


def self_flops(H: int, D: int, lens) -> int:
    """Self-attention of every user sequence over itself: 4·H·D·Σ_u L_u²."""
    return 4 * H * D * sum(int(L) * int(L) for L in lens)


def self_extra_bytes(H: int, D: int, T: int) -> int:
    """What fusing the self-attention adds to the algorithmic bytes: q_user read and
    out_user written once (its K/V are the target attention's, read once for both)."""
    return 2 * T * H * D * BF16


def workload_numbers(wl) -> dict:
    """FLOPs, algorithmic bytes and the broadcast path's extra bytes of a workload."""
    c = wl.cfg
    return {
        "flops": flops(c.H, c.D, c.Lq, wl.S),
        "alg_bytes": alg_bytes(c.H, c.D, c.Lq, wl.T, wl.n_cand, wl.n_user),
        "broadcast_extra_bytes": broadcast_extra_bytes(c.H, c.D, wl.S),
    }


# ----------------------------------------------------------------------------- linear compression

def gemm_intensity(B: int, M: int, K: int, N: int, elem_bytes: int = BF16) -> float:
    """FLOP/B of the batched product (M, K) @ (B, K, N) -> (B, M, N): 2·B·M·K·N over the
    shared A read once plus every batch entry's B read and C written once ("In-Kernel
    Broadcast Optimization", Appendix 2; the broadcast form of linear compression, §2)."""
    return 2 * B * M * K * N / ((M * K + B * K * N + B * M * N) * elem_bytes)


def lce_flops(M: int, N: int, n_user: int, K_user: int, n_cand: int, K_cand: int) -> int:
    """The decomposed work (§2.1): the user product at the user batch size, the candidate
    product at the candidate batch size; 2 FLOPs per multiply-add, unpadded K."""
    return 2 * M * N * (n_user * K_user + n_cand * K_cand)


def lce_alg_bytes(M: int, N: int, n_user: int, Kp_user: int, n_cand: int, Kp_cand: int) -> int:
    """What the two launches must move, with K padded as the kernel reads it: both weight
    blocks and every X block read once, the bf16 user term written once and read once,
    the bf16 output written once, the int32 candidate map."""
    w = M * (Kp_user + Kp_cand) * BF16
    x = (n_user * Kp_user + n_cand * Kp_cand) * N * BF16
    term = 2 * n_user * M * N * BF16
    out = n_cand * M * N * BF16
    return w + x + term + out + 4 * n_cand


def ml_lce_flops(M: int, N: int, n_user: int, K_user: int, n_vendor: int, K_vendor: int,
                 n_item: int, K_item: int) -> int:
    """Three levels (§5), each product at its own batch size."""
    return 2 * M * N * (n_user * K_user + n_vendor * K_vendor + n_item * K_item)


def ml_lce_alg_bytes(M: int, N: int, n_user: int, Kp_user: int, n_vendor: int, Kp_vendor: int,
                     n_item: int, Kp_item: int) -> int:
    """Three launches: W and X of every level read once, the bf16 user and vendor terms
    each written once and read once, the bf16 output, the two int32 maps."""
    w = M * (Kp_user + Kp_vendor + Kp_item) * BF16
    x = (n_user * Kp_user + n_vendor * Kp_vendor + n_item * Kp_item) * N * BF16
    terms = 2 * (n_user + n_vendor) * M * N * BF16
    out = n_item * M * N * BF16
    return w + x + terms + out + 4 * (n_item + n_vendor)
