"""The bench's FLOP and byte accounting, pinned to the numbers the IKBO pages print."""
import json
import os

from broadcast_target_attention_gb300 import accounting as A
from broadcast_target_attention_gb300 import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def test_arithmetic_intensity_matches_pages():
    with open(os.path.join(HERE, "golden", "ai_closed_form.json")) as f:
        g = json.load(f)
    s = g["setting"]
    std = A.ai_per_user_head(1, s["n_seed_queries_per_candidate"], s["user_seq_len"])
    ikbo = A.ai_per_user_head(s["candidates_per_user"], s["n_seed_queries_per_candidate"],
                              s["user_seq_len"])
    assert abs(std - g["standard_flop_per_byte"]) < 0.6
    assert abs(ikbo - g["ikbo_flop_per_byte"]) < 0.6


def test_intensity_from_flops_and_bytes():
    """ai_per_user_head is flops / bytes of one user-head, indices aside."""
    r, Lq, L, D = 70, 64, 1024, 128
    fl = A.flops(1, D, Lq, r * L)
    by = A.alg_bytes(1, D, Lq, L, r, 1) - 4 * (r + 2)
    assert abs(fl / by - A.ai_per_user_head(r, Lq, L)) < 1e-9


def test_headline_workload_numbers():
    wl = W.generate(W.CONFIGS[W.HEADLINE])
    n = A.workload_numbers(wl)
    assert n["flops"] == 4 * 4 * 128 * 1 * wl.S
    # 1024 candidates / 15 users, L in [256, 1024], H=4, D=128: ~21-22 MB of algorithmic traffic
    assert 18e6 < n["alg_bytes"] < 24e6


# ----------------------------------------------------------------------------- linear compression

def test_lce_broadcast_intensity_matches_pages():
    with open(os.path.join(HERE, "golden", "lce_intensity.json")) as f:
        g = json.load(f)
    s = g["setting"]
    ai = A.gemm_intensity(s["B"], s["M"], s["K"], s["N"], s["bytes_per_element"])
    assert g["broadcast_gemm_flop_per_byte"] <= ai < g["broadcast_gemm_flop_per_byte"] + 1


def _counted_flops(*products):
    """FLOPs of the given (W, X) batched products as torch's own FLOP counter sees them."""
    import torch
    from torch.utils.flop_counter import FlopCounterMode
    with FlopCounterMode(display=False) as fc:
        for Wt, Xt in products:
            torch.matmul(Wt, Xt)
    return fc.get_total_flops()


def test_lce_numbers_against_the_tensors():
    """FLOPs: torch's counter over the two decomposed products at their own batch sizes.
    Bytes: the generated tensors' own sizes, plus the term written and read back once and
    the output written once."""
    import torch
    cfg = W.LceConfig(name="a", n_cand=9, n_user=4, M=37, K_user=13, K_cand=21, N=64, seed=1)
    wl = W.lce_generate(cfg)
    unpadded = [(torch.zeros(cfg.M, cfg.K_user), torch.zeros(cfg.n_user, cfg.K_user, cfg.N)),
                (torch.zeros(cfg.M, cfg.K_cand), torch.zeros(cfg.n_cand, cfg.K_cand, cfg.N))]
    assert A.lce_flops(cfg.M, cfg.N, cfg.n_user, cfg.K_user, cfg.n_cand, cfg.K_cand) == \
        _counted_flops(*unpadded)
    ku, kc = wl.X_user.shape[1], wl.X_cand.shape[1]
    assert ku % 8 == 0 and kc % 8 == 0 and ku >= cfg.K_user and kc >= cfg.K_cand
    term = cfg.n_user * cfg.M * cfg.N * 2
    out = cfg.n_cand * cfg.M * cfg.N * 2
    want = sum(a.nbytes for a in (wl.W_user, wl.W_cand, wl.X_user, wl.X_cand, wl.cand_to_user)) \
        + 2 * term + out
    assert A.lce_alg_bytes(cfg.M, cfg.N, cfg.n_user, ku, cfg.n_cand, kc) == want


def test_ml_lce_numbers_against_the_tensors():
    import torch
    cfg = W.LceMlConfig(name="a", n_item=11, n_vendor=5, n_user=2, M=19, K_user=13, K_vendor=9,
                        K_item=21, N=64, seed=2, shuffle=True)
    l = W.lce_ml_generate(cfg)
    products = [(torch.zeros(cfg.M, k), torch.zeros(n, k, cfg.N))
                for n, k in ((cfg.n_user, cfg.K_user), (cfg.n_vendor, cfg.K_vendor),
                             (cfg.n_item, cfg.K_item))]
    assert A.ml_lce_flops(cfg.M, cfg.N, cfg.n_user, cfg.K_user, cfg.n_vendor, cfg.K_vendor,
                          cfg.n_item, cfg.K_item) == _counted_flops(*products)
    ku, kv, ki = l.X_user.shape[1], l.X_vendor.shape[1], l.X_item.shape[1]
    terms = (cfg.n_user + cfg.n_vendor) * cfg.M * cfg.N * 2
    out = cfg.n_item * cfg.M * cfg.N * 2
    want = sum(a.nbytes for a in (l.W_user, l.W_vendor, l.W_item, l.X_user, l.X_vendor, l.X_item,
                                  l.item_to_vendor, l.vendor_to_user)) + 2 * terms + out
    # the bench counts the item map and one int32 per vendor (its user), as the kernels read them
    assert A.ml_lce_alg_bytes(cfg.M, cfg.N, cfg.n_user, ku, cfg.n_vendor, kv, cfg.n_item, ki) == want


def test_decomposition_cuts_the_user_side_work_by_the_ratio():
    """§2.1: at ~70 candidates per user the user-side product shrinks ~70x; the candidate side
    is unchanged."""
    with open(os.path.join(HERE, "golden", "lce_intensity.json")) as f:
        g = json.load(f)
    B, M, K, N = (g["setting"][k] for k in ("B", "M", "K", "N"))
    Ku = K // 2
    broadcast = A.lce_flops(M, N, B, Ku, B, K - Ku)          # every candidate its own user block
    ikbo = A.lce_flops(M, N, g["B_user"], Ku, B, K - Ku)
    user_ratio = (broadcast - A.lce_flops(M, N, 0, Ku, B, K - Ku)) / \
        (ikbo - A.lce_flops(M, N, 0, Ku, B, K - Ku))
    assert abs(user_ratio - B / g["B_user"]) < 1e-9
    assert 60 < user_ratio < 80
