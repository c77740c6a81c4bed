"""Writes tests/golden/oracle_tiny_rows.json from the fp64 oracle alone.

The pages print no worked numeric example of attention or of the merge, so
the stored values here are the oracle's own, on the seeded tiny non-causal
workload (B=1, H=2, S=256, D=64) and on the same inputs under causal
masking, for a few query rows per head. They pin the oracle against
accidental change and give the GPU tests a fixed expected value.

Run:  python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
import workloads  # noqa: E402

ROWS = [0, 1, 127, 128, 200, 255]


def main():
    w = workloads.WORKLOADS["tiny_b1h2s256d64"]
    q, k, v = workloads.make_qkv(w)
    rows = np.array([ROWS] * (w.B * w.Hq), dtype=np.int64)
    out = {"workload": w.name, "seed": w.seed, "rows": ROWS, "cases": {}}
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal, rows=rows, threads=1)
        out["cases"]["causal" if causal else "noncausal"] = {
            "o": [[[float.hex(float(x)) for x in r] for r in h] for h in o[0]],
            "lse": [[float.hex(float(x)) for x in h] for h in lse[0]],
        }
    with open(os.path.join(HERE, "oracle_tiny_rows.json"), "w") as f:
        json.dump(out, f, indent=0)


if __name__ == "__main__":
    main()
