"""Every planted mistake in the oracle must be caught by at least one pin.

Each mutant is oracle.c compiled with -DORC_MUTANT=k (see the mutant list at
the top of oracle.c): dropped log-weight term, wrong sign of the cost, weights
transposed, gradient missing a_i, wrong sign of g in the plan, Jacobi instead
of Gauss-Seidel order, log-sum-exp without the max added back, a coordinate
dropped from the cost, a cosine cost that leaves y unnormalised, a transport
product that weights its pairs with the wrong row weight, a sparse APML that drops
the column softmax, a Hessian-vector product that holds the column potentials
fixed, a COO threshold with the sign of log tau flipped, a COO row test made
against a column maximum.
"""
import pytest

import oracle_pins
from oracle import oracle as O

MUTANTS = {1: "drops log b", 2: "sign of C", 3: "weights transposed", 4: "grad without a_i",
           5: "sign of g in plan", 6: "Jacobi order", 7: "LSE without max", 8: "cost drops a coordinate",
           9: "cosine without y normalised", 10: "transport with the wrong row weight",
           11: "APML without the column softmax", 12: "HVP with the column potentials fixed",
           13: "COO threshold with the sign of log tau flipped", 14: "COO row test against the column maximum"}


@pytest.mark.parametrize("k", sorted(MUTANTS), ids=lambda k: MUTANTS[k])
def test_mutant_is_caught(k, tmp_path):
    orc = O.Oracle(O.build(mutant=k, out_dir=str(tmp_path)))
    assert orc.mutant == k
    caught = []
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(orc)
        except (AssertionError, FloatingPointError, ValueError, RuntimeError) as e:
            caught.append((pin.__name__, str(e)[:80]))
            break
    assert caught, f"mutant {k} ({MUTANTS[k]}) passed every pin"
