"""Writes tests/golden/tiny_8x2.json from the oracle alone (no CUDA code involved).

Run from the repository root:  python tests/golden/make_golden.py
"""
import hashlib
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from broadcast_target_attention_gb300 import workloads as W  # noqa: E402


def main():
    wl = W.generate(W.CONFIGS["tiny_8x2"])
    out = oracle.attention_wl(wl)
    rows = []
    for c in (0, 4, 5, 7):
        for h in (0, 1):
            rows.append({"c": c, "h": h, "out0_8": [float(x) for x in out[c, h, 0, :8]]})
    doc = {
        "what": "oracle output of the tiny configuration (2 users, 8 candidates, L=16/24, "
                "H=2, D=64, Lq=1, seed 0): first 8 values of selected rows",
        "inputs_sha256": hashlib.sha256(wl.q.tobytes() + wl.k.tobytes() + wl.v.tobytes()).hexdigest(),
        "rows": rows,
    }
    path = os.path.join(ROOT, "tests", "golden", "tiny_8x2.json")
    with open(path, "w") as f:
        json.dump(doc, f, indent=1)
        f.write("\n")


if __name__ == "__main__":
    main()
