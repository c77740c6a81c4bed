"""The oracle reproduces its stored values bit for bit (tests/golden/make_golden.py)."""
import json
import os

import numpy as np

import oracle
import workloads

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "oracle_tiny_rows.json")


def load_golden():
    with open(GOLDEN) as f:
        g = json.load(f)
    cases = {}
    for name, c in g["cases"].items():
        o = np.array([[[float.fromhex(x) for x in r] for r in h] for h in c["o"]])
        lse = np.array([[float.fromhex(x) for x in h] for h in c["lse"]])
        cases[name] = (o, lse)
    return g, cases


def test_oracle_matches_stored_values():
    g, cases = load_golden()
    w = workloads.WORKLOADS[g["workload"]]
    q, k, v = workloads.make_qkv(w)
    rows = np.array([g["rows"]] * (w.B * w.Hq), dtype=np.int64)
    for name, (o_ref, lse_ref) in cases.items():
        o, lse = oracle.attention(q, k, v, name == "causal", rows=rows, threads=3)
        np.testing.assert_allclose(o[0], o_ref, rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[0], lse_ref, rtol=0, atol=1e-14)
