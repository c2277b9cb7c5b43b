"""Writes the exact fixtures of this folder.  Calls only ``oracle.exact``.

Each fixture is a small integer/rational example whose expected outputs are the
exact pair sum of the masked second-order output (page "Higher-order Linear
Attention", technical summary, item "1. Zweite Ordnung HLA"; section summary §2.1,
§4.3), stored as exact fractions "p/q".  Inputs are small integers chosen by hand
so that every pair weight is distinct.

Run:  python tests/golden/make_golden.py
"""
from __future__ import annotations

import json
import os
import sys
from fractions import Fraction

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle.exact import pair_sum  # noqa: E402

CASES = {
    # n = 2, d = dv = 1: the two-token closed form, decay 1/2
    "n2_d1": {
        "q": [[1], [2]], "k": [[1], [3]], "v": [[1], [-2]], "gamma": "1/2",
    },
    # n = 5, d = 2, dv = 3, decay 3/4: every (i, j, t) weight different
    "n5_d2": {
        "q": [[1, 0], [2, -1], [0, 1], [1, 1], [-1, 2]],
        "k": [[1, 2], [0, 1], [3, -1], [1, 0], [2, 2]],
        "v": [[1, 0, -1], [2, 1, 0], [0, -3, 1], [1, 1, 1], [-2, 0, 4]],
        "gamma": "3/4",
    },
    # n = 4, d = 3, dv = 2, no decay
    "n4_d3_nodecay": {
        "q": [[1, -1, 0], [0, 2, 1], [1, 1, 1], [-1, 0, 2]],
        "k": [[2, 0, 1], [1, 1, -1], [0, -2, 1], [1, 0, 0]],
        "v": [[1, 2], [-1, 0], [3, 1], [0, -2]],
        "gamma": "1",
    },
}


def main():
    for name, case in CASES.items():
        F = lambda rows: [[Fraction(x) for x in r] for r in rows]  # noqa: E731
        o, den = pair_sum(F(case["q"]), F(case["k"]), F(case["v"]), Fraction(case["gamma"]))
        doc = {
            "source": "exact pair sum of the masked second-order output; page "
                      "'Higher-order Linear Attention', technical summary item "
                      "'1. Zweite Ordnung HLA' (o_t = q_t^T(S_t C_t - G_t)), section "
                      "summary §2.1 (mask j <= t) and §4.3 (fixed decay)",
            "writer": "tests/golden/make_golden.py (oracle.exact.pair_sum)",
            **case,
            "out": [[str(x) for x in row] for row in o],
            "den": [str(x) for x in den],
        }
        with open(os.path.join(HERE, f"{name}.json"), "w") as f:
            json.dump(doc, f, indent=1)
            f.write("\n")


if __name__ == "__main__":
    main()
