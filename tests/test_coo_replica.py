"""The fp32 COO replica (a test checker) against a support worked by hand (CPU).

The problem is the 3 x 3 one of ``oracle_pins.pin_coo_threshold_hand_worked``
("CUDA-Optimized APML", Abstract / Innovation: the support keeps the pairs
within a factor tau of their row's, or column's, largest entry).  Its ratios
to the row and column maxima are 7 % or more away from every tau used, so
fp32 rounding cannot move a decision and the replica must list exactly the
hand-worked supports, in both of the library's layouts.
"""
import numpy as np
import pytest

import coo_replica

LN2 = np.log(2.0)
X = np.array([[0.0], [1.0], [3.0]])
Y = np.array([[0.0], [2.0], [5.0]])
A = np.array([0.5, 0.25, 0.25])
Bw = np.array([0.25, 0.25, 0.5])
F = np.zeros(3)
G = np.array([0.0, 1.0, 0.0])
CASES = [
    (0.03, 1, [(0, 0), (0, 1), (1, 0), (1, 1), (2, 1), (2, 2)]),
    (0.04, 1, [(0, 0), (0, 1), (1, 0), (1, 1), (2, 1)]),
    (0.06, 1, [(0, 0), (1, 0), (1, 1), (2, 1)]),
    (0.06, 2, [(0, 0), (0, 1), (1, 0), (1, 1), (2, 1), (2, 2)]),
    (0.15, 2, [(0, 0), (1, 0), (1, 1), (2, 1), (2, 2)]),
    (0.20, 2, [(0, 0), (1, 1), (2, 1), (2, 2)]),
    (0.15, 3, [(0, 0), (1, 0), (1, 1), (2, 1), (2, 2)]),
]


def _operands(d):
    """Operands in the library's layout for eps = 1: the point layout (d <= 3)
    holds L = kappa (0 - f); the dense layout (d > 3) holds L = kappa (|x|^2 - f),
    which shifts every score of a row (column) by the same constant."""
    kappa = np.float32(1.0 / LN2)
    xc = np.zeros((3, d), np.float32)
    yc = np.zeros((3, d), np.float32)
    xc[:, 0], yc[:, 0] = X[:, 0], Y[:, 0]
    nx = (xc.astype(np.float64) ** 2).sum(1) if d > 3 else np.zeros(3)
    ny = (yc.astype(np.float64) ** 2).sum(1) if d > 3 else np.zeros(3)
    Lx = (kappa * (nx - F)).astype(np.float32)
    Ly = (kappa * (ny - G)).astype(np.float32)
    return xc, np.log2(A).astype(np.float32), Lx, yc, np.log2(Bw).astype(np.float32), Ly, float(kappa)


@pytest.mark.parametrize("d", [1, 3, 4, 8])
@pytest.mark.parametrize("tau,dirs,want", CASES)
def test_replica_hand_worked_support(d, tau, dirs, want):
    xc, lwx, Lx, yc, lwy, Ly, kappa = _operands(d)
    got = coo_replica.replica(xc, lwx, Lx, yc, lwy, Ly, kappa, float(np.float32(np.log2(tau))), dirs)
    pairs = list(zip(got["rows"].tolist(), got["cols"].tolist()))
    assert pairs == want


def test_replica_maxima_and_limits():
    xc, lwx, Lx, yc, lwy, Ly, kappa = _operands(1)
    full = coo_replica.replica(xc, lwx, Lx, yc, lwy, Ly, kappa, -np.inf, 3)
    assert len(full["rows"]) == 9, "log2 tau = -inf keeps every pair"
    top = coo_replica.replica(xc, lwx, Lx, yc, lwy, Ly, kappa, 0.0, 1)
    assert list(zip(top["rows"].tolist(), top["cols"].tolist())) == [(0, 0), (1, 1), (2, 1)]
    # row maxima in log2 units: max_j kappa (g_j - C_ij) + log2 b_j, worked by hand
    want = np.array([np.log2(0.25), np.log2(0.25), np.log2(0.25)])
    assert np.allclose(full["Mr"], want, rtol=0, atol=1e-6)
