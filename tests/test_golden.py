"""The oracle still computes what tests/golden/oracle_regression.json holds
(written by tests/golden/make_golden.py from oracle/ alone): a guard against
an unintended change of the oracle's arithmetic, not a correctness pin."""

import json
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.join(HERE, "golden"))

import make_golden  # noqa: E402


def test_oracle_matches_stored_values():
    with open(os.path.join(HERE, "golden", "oracle_regression.json")) as f:
        stored = json.load(f)
    now = make_golden.cases()
    assert set(stored) == set(now)
    for case, outs in stored.items():
        for k, v in outs.items():
            np.testing.assert_allclose(now[case][k], np.array(v), rtol=1e-12, atol=1e-15, err_msg=f"{case} {k}")
