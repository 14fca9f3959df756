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
