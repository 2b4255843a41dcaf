"""Writes tests/golden/oracle_q128_kv256.txt from the FP64 oracle alone.

The stored values guard the oracle against unintended change: for the seeded
128-token chunk at the end of a 256-key prefix (24 query heads, 4 KV heads,
head_dim 256, scale 1/16), selected rows' LSE and a few output columns.
Run: python tests/golden/make_golden.py
"""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gqa_inputs import WORKLOADS, make_workload  # noqa: E402

ROWS = [0, 5, 23, 24 * 64 + 7, 24 * 127 + 23]
COLS = [0, 1, 128, 255]


def main():
    w = WORKLOADS["q128_kv256"]
    q, k, v = make_workload(w)
    out, lse = oracle.attention(q, k, v, w.scale, rows=ROWS)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_q128_kv256.txt")
    with open(path, "w") as f:
        f.write("# FP64 oracle, workload q128_kv256 (seed 1000), written by make_golden.py\n")
        f.write("# row_id lse out[c] for c in " + " ".join(map(str, COLS)) + "\n")
        for i, r in enumerate(ROWS):
            vals = " ".join(f"{out[i, c]:.17g}" for c in COLS)
            f.write(f"{r} {lse[i]:.17g} {vals}\n")


if __name__ == "__main__":
    main()
