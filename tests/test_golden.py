"""Regression guard: the oracle reproduces its committed outputs for two tiny seeded cases."""
import json
import os

import numpy as np

from tests.golden.make_golden import compute

HERE = os.path.dirname(os.path.abspath(__file__))


def test_oracle_matches_committed_golden():
    with open(os.path.join(HERE, "golden", "oracle_tiny.json")) as f:
        doc = json.load(f)
    for case in doc["cases"]:
        o, S = compute(case)
        np.testing.assert_allclose(o.ravel(), np.array(case["o"]), rtol=1e-14, atol=1e-15)
        np.testing.assert_allclose(S.ravel(), np.array(case["S_T"]), rtol=1e-14, atol=1e-15)
