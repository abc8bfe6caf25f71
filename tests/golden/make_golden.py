"""Writes tests/golden/oracle_tiny.json: oracle outputs for two tiny seeded cases.

The values come from ``oracle.forward`` only (the float64 recurrence of the Kev-4B-LiteRT page
"r15_kernel_test.py", truth_f64); they guard the oracle against unintended changes. Inputs are
regenerated from their seeds by ``gated_deltanet_rule_gb300.inputs.regime``.
Run: python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from gated_deltanet_rule_gb300 import inputs  # noqa: E402

CASES = [
    {"name": "R1", "L": 6, "seed": 11, "Hk": 1, "Hv": 2, "Dk": 4, "init_state": True, "n_valid": None},
    {"name": "R3", "L": 7, "seed": 32, "Hk": 1, "Hv": 2, "Dk": 4, "init_state": True, "n_valid": 5},
]


def compute(case):
    x = inputs.regime(case["name"], case["L"], case["seed"], Hk=case["Hk"], Hv=case["Hv"],
                      Dk=case["Dk"], init_state=case["init_state"], n_valid=case["n_valid"])
    o, S = oracle.forward(x.q, x.k, x.v, x.g, x.beta, x.S0)
    return o, S


if __name__ == "__main__":
    out = {"source": "oracle.forward (float64 token recurrence)", "cases": []}
    for c in CASES:
        o, S = compute(c)
        out["cases"].append({**c, "o": o.ravel().tolist(), "S_T": S.ravel().tolist()})
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "oracle_tiny.json")
    with open(path, "w") as f:
        json.dump(out, f, indent=0)
    print(path)
