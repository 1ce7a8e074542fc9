"""Writes tests/golden/oracle_regression.json: float64 oracle outputs on three
tiny seeded problems (the scan, its gradients, the generalised scan with the
zero-order hold), from oracle/ alone.

The pages print no worked numerical example, so no stored value here comes
from them. These values do not pin the oracle's correctness (the pins in
tests/pins.py do that); they catch an unintended change of its arithmetic.
A change that is intended rewrites the file by running this script and names,
in its commit message, the passage or reading that justifies it.

    python tests/golden/make_golden.py
"""

import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from workloads import gen  # noqa: E402


def cases():
    x = gen.random_scan_inputs(1, 6, 3, 4, in_dtype="f32", seed=101, with_h0=True, a_log_jitter=0.3)
    y, h = oracle.scan(x)
    dy, dh = gen.random_output_grads(1, 6, 3, 4, "f32", seed=102)
    g = oracle.scan_bwd(x, dy, dh)
    xg = gen.random_general_inputs(1, 5, 4, 16, 2, in_dtype="bf16", seed=103, with_h0=True)
    yg, hg = oracle.scan_general(xg, 2, "zoh")
    return {
        "scan_1x6x3_n4_f32_seed101": {"y": y.tolist(), "h_last": h.tolist()},
        "scan_bwd_1x6x3_n4_f32_seed101_dy102": {k: v.tolist() for k, v in g.items()},
        "general_zoh_1x5x4_n16_g2_bf16_seed103": {"y": yg.tolist(), "h_last": hg.tolist()},
    }


if __name__ == "__main__":
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as f:
        json.dump(cases(), f, indent=None, separators=(",", ":"))
    print("written")
