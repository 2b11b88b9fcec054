"""Writes two_point.json: 2 x 2 entropic OT problems with their exact plans.

The expected values come from the closed form of a 2 x 2 Sinkhorn plan, not
from any solver: a plan with marginals (a, b) is P = [[p, a1-p], [b1-p, a2-b1+p]],
and a Sinkhorn plan diag(u) K diag(v), K = exp(-C/eps), has the cross ratio
P11 P22 / (P12 P21) = K11 K22 / (K12 K21); that fixes p as the feasible root of
a quadratic (see ``two_point_plan`` in tests/oracle_pins.py).  The cost and the
gradient follow from P by their definitions:
cost = sum_ij P_ij C_ij, grad_i = 2 (a_i x_i - sum_j P_ij y_j).

Run:  python tests/golden/make_two_point.py
"""
import json
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
from oracle_pins import two_point_plan  # noqa: E402  (closed form only)

CASES = [
    # X, Y, a, b, eps
    ([[0.0, 0.0], [1.0, 0.2]], [[0.9, 0.1], [0.1, -0.3]], [0.3, 0.7], [0.6, 0.4], 0.5),
    ([[0.2, 0.5, -0.1], [-0.4, 0.3, 0.8]], [[0.1, 0.1, 0.1], [-0.5, 0.6, 0.4]], [0.55, 0.45], [0.2, 0.8], 0.1),
    ([[1.0], [2.0]], [[1.5], [0.0]], [0.5, 0.5], [0.5, 0.5], 2.0),
]


def main():
    out = []
    for X, Y, a, b, eps in CASES:
        Xa, Ya = np.array(X), np.array(Y)
        C = ((Xa[:, None, :] - Ya[None, :, :]) ** 2).sum(-1)
        P = two_point_plan(C, a, b, eps)
        cost = float((P * C).sum())
        grad = 2 * (np.array(a)[:, None] * Xa - P @ Ya)
        out.append(dict(X=X, Y=Y, a=a, b=b, eps=eps, iters=4000, P=P.tolist(), cost=cost,
                        grad=grad.tolist()))
    doc = dict(source="closed form of the 2 x 2 entropic plan (cross-ratio identity); "
                      "written by tests/golden/make_two_point.py", cases=out)
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "two_point.json")
    with open(path, "w") as fh:
        json.dump(doc, fh, indent=1)
    print("wrote", path)


if __name__ == "__main__":
    main()
