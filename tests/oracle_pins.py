"""Pins of the fp64 oracle against facts that do not come from the oracle.

Each ``pin_*`` takes an :class:`oracle.oracle.Oracle` and raises
``AssertionError`` when the oracle disagrees with a closed form, a textbook
special case, an invariance or brute force.  ``test_oracle_pins.py`` runs them
against the real oracle; ``test_oracle_mutants.py`` runs them against builds of
the oracle with a planted mistake and checks that every mistake is caught.

The pages ("FlashSinkhorn", Methodologie 1-3; "CUDA-Optimized APML",
Abstract) print no worked numeric example, so these pins replace one.
"""
from __future__ import annotations

import itertools
import json
import os

import numpy as np
from scipy.special import logsumexp

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, rtol, atol=0.0, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    err = np.max(np.abs(a - b)) if a.size else 0.0
    lim = atol + rtol * max(np.max(np.abs(b)) if b.size else 0.0, 1e-300)
    assert err <= lim, f"{what}: max|diff| {err:.3e} > {lim:.3e}"


def _gauge(f, g, fr, gr):
    """Remove the common constant shift (f + c, g - c) before comparing."""
    c = 0.5 * (np.mean(f - fr) - np.mean(g - gr))
    return f - c, g + c


def pin_closed_form_single_point(orc):
    """n = m = 1, a = b = 1: after any number of iterations f = |x-y|^2, g = 0,
    cost = |x-y|^2 and grad = 2(x - y)."""
    rng = _rng(1)
    for d in (1, 3, 5):
        x = rng.normal(size=(1, d))
        y = rng.normal(size=(1, d))
        c = float(np.sum((x - y) ** 2))
        for eps, it in ((0.01, 1), (0.5, 4)):
            f, g = orc.sinkhorn(x, y, [1.0], [1.0], [eps], [it])
            _close(f, [c], 1e-12, what="f at n=1")
            _close(g, [0.0], 0, atol=1e-12 * c, what="g at n=1")
            out = orc.plan_apply(x, y, [1.0], [1.0], f, g, eps)
            _close(out["cost"], c, 1e-12, what="cost at n=1")
            _close(out["grad"], 2 * (x - y), 1e-12, what="grad at n=1")


def two_point_plan(C, a, b, eps):
    """Exact entropic plan of a 2 x 2 problem.

    P = [[p, a1 - p], [b1 - p, a2 - b1 + p]] has the right marginals for any p,
    and a Sinkhorn plan diag(u) K diag(v) satisfies
    P11 P22 / (P12 P21) = K11 K22 / (K12 K21) = rho = exp(-(C11 + C22 - C12 - C21)/eps),
    which is a quadratic in p with one root in the feasible interval.
    """
    a1, a2 = a
    b1, _ = b
    rho = np.exp(-(C[0, 0] + C[1, 1] - C[0, 1] - C[1, 0]) / eps)
    A = 1.0 - rho
    Bq = a2 - b1 + rho * (a1 + b1)
    Cq = -rho * a1 * b1
    lo, hi = max(0.0, b1 - a2), min(a1, b1)
    if abs(A) < 1e-14:
        roots = [-Cq / Bq]
    else:
        disc = np.sqrt(Bq * Bq - 4 * A * Cq)
        # numerically stable pair of roots
        q = -0.5 * (Bq + np.copysign(disc, Bq))
        roots = [q / A, Cq / q]
    p = [r for r in roots if lo - 1e-15 <= r <= hi + 1e-15]
    assert len(p) >= 1, "no feasible root"
    p = p[0]
    return np.array([[p, a1 - p], [b1 - p, a2 - b1 + p]])


def pin_two_point_closed_form(orc):
    """2 x 2 problems with unequal weights converge to the closed-form plan."""
    with open(os.path.join(GOLDEN, "two_point.json")) as fh:
        cases = json.load(fh)["cases"]
    for case in cases:
        X = np.array(case["X"])
        Y = np.array(case["Y"])
        a = np.array(case["a"])
        b = np.array(case["b"])
        eps = case["eps"]
        f, g = orc.sinkhorn(X, Y, a, b, [eps], [case["iters"]])
        out = orc.plan_apply(X, Y, a, b, f, g, eps)
        P = np.array(case["P"])
        _close(out["rowsum"], P.sum(1), 1e-10, what="2x2 row sums")
        _close(out["cost"], case["cost"], 1e-10, what="2x2 cost")
        _close(out["grad"], np.array(case["grad"]), 1e-9, what="2x2 grad")


def pin_attention_form(orc):
    """Propositie 1 ("FlashSinkhorn", Methodologie 1): with Q = sqrt2 X,
    K = sqrt2 Y, g_hat = g - |y|^2, delta = eps log b, the f-half equals
    |x_i|^2 - eps * LSE_j[(Q K^T + 1 (g_hat + delta)^T)/eps]; the g-half is the
    mirror with f_hat = f - |x|^2 and gamma = eps log a.  Evaluated here in the
    expanded (dot-product) form, against the oracle's direct form."""
    rng = _rng(2)
    n, m, d = 37, 29, 4
    X = rng.normal(size=(n, d))
    Y = rng.normal(size=(m, d)) + 0.3
    a = rng.random(n) + 0.1
    a /= a.sum()
    b = rng.random(m) + 0.1
    b /= b.sum()
    g = rng.normal(size=m)
    f = rng.normal(size=n)
    for eps in (0.05, 1.0):
        Q, K = np.sqrt(2) * X, np.sqrt(2) * Y
        S = (Q @ K.T + (g - (Y * Y).sum(1) + eps * np.log(b))[None, :]) / eps
        f_att = (X * X).sum(1) - eps * logsumexp(S, axis=1)
        _close(orc.f_half(X, Y, b, g, eps), f_att, 1e-11, atol=1e-11, what="attention form, f-half")
        S2 = (K @ Q.T + (f - (X * X).sum(1) + eps * np.log(a))[None, :]) / eps
        g_att = (Y * Y).sum(1) - eps * logsumexp(S2, axis=1)
        _close(orc.g_half(X, Y, a, f, eps), g_att, 1e-11, atol=1e-11, what="attention form, g-half")


def _problem(seed, n, m, d, scale=1.0):
    rng = _rng(seed)
    X = scale * rng.normal(size=(n, d))
    Y = scale * rng.normal(size=(m, d)) + 0.2
    a = rng.random(n) + 0.2
    a /= a.sum()
    b = rng.random(m) + 0.2
    b /= b.sum()
    return X, Y, a, b


def pin_marginals_and_duality(orc):
    """At convergence the plan has both marginals, and the dual objective
    <a,f> + <b,g> equals <C,P> + eps KL(P || a x b)."""
    X, Y, a, b = _problem(3, 23, 17, 2)
    eps = 0.2
    f, g = orc.sinkhorn(X, Y, a, b, [eps], [1500])
    out = orc.plan_apply(X, Y, a, b, f, g, eps)
    assert np.abs(out["rowsum"] - a).sum() < 1e-10, "row marginal not reached"
    assert np.abs(out["colsum"] - b).sum() < 1e-12, "column marginal not exact after a g-half"
    dual, primal = orc.objectives(X, Y, a, b, f, g, eps)
    _close(dual, primal, 1e-9, what="duality")


def pin_brute_force_assignment(orc):
    """Uniform clouds with n = m <= 6: 0 <= <C,P_eps> - OT_0 <= eps log n, with
    OT_0 the best permutation found by enumeration; at small eps the row argmax
    of the plan is that permutation."""
    rng = _rng(4)
    for n in (3, 5, 6):
        for trial in range(3):
            X = rng.random((n, 2))
            Y = rng.random((n, 2))
            C = ((X[:, None, :] - Y[None, :, :]) ** 2).sum(-1)
            costs = sorted((np.mean(C[np.arange(n), list(p)]), p) for p in itertools.permutations(range(n)))
            ot0, best = costs[0]
            gap = costs[1][0] - ot0
            for eps in (0.05, 0.01):
                f, g = orc.sinkhorn(X, Y, None, None, [eps], [3000])
                out = orc.plan_apply(X, Y, None, None, f, g, eps)
                slack = np.abs(out["rowsum"] - 1.0 / n).sum() * C.max()
                assert out["cost"] >= ot0 - slack - 1e-12, "entropic cost below the exact OT cost"
                assert out["cost"] <= ot0 + eps * np.log(n) + slack + 1e-12, "entropic cost above OT_0 + eps log n"
            if gap > 0.02:
                epss = [0.1, 0.03, 0.01, 0.003, 1e-3]
                f, g = orc.sinkhorn(X, Y, None, None, epss, [400] * len(epss))
                eps = epss[-1]
                a = np.full(n, 1.0 / n)
                s = (f[:, None] + g[None, :] - C) / eps
                assert tuple(np.argmax(s, axis=1)) == tuple(best), "argmax of the plan is not the optimal permutation"


def pin_sorted_matching_1d(orc):
    """d = 1, uniform weights: the exact OT cost is the sorted (monotone)
    matching; the entropic cost lies within eps log n above it."""
    rng = _rng(5)
    n = 96
    x = rng.random(n)
    y = rng.random(n) * 0.8 + 0.3
    ot0 = np.mean((np.sort(x) - np.sort(y)) ** 2)
    for eps in (0.02, 0.005):
        f, g = orc.sinkhorn(x[:, None], y[:, None], None, None, [eps * 4, eps * 2, eps], [200, 200, 600])
        out = orc.plan_apply(x[:, None], y[:, None], None, None, f, g, eps)
        slack = np.abs(out["rowsum"] - 1.0 / n).sum()
        assert ot0 - slack - 1e-12 <= out["cost"] <= ot0 + eps * np.log(n) + slack + 1e-12, \
            f"1-D sorted matching bound violated: {out['cost']} vs {ot0}"


def pin_large_eps(orc):
    """eps -> infinity: P -> a x b, so cost -> sum_i a_i|x_i|^2 + sum_j b_j|y_j|^2
    - 2 xbar_a . ybar_b and grad_i -> 2 a_i (x_i - ybar_b), errors O(Var C / eps)."""
    X, Y, a, b = _problem(6, 31, 27, 3)
    eps = 1e6
    f, g = orc.sinkhorn(X, Y, a, b, [eps], [3])
    out = orc.plan_apply(X, Y, a, b, f, g, eps)
    xb = a @ X
    yb = b @ Y
    c_inf = a @ (X * X).sum(1) + b @ (Y * Y).sum(1) - 2 * xb @ yb
    _close(out["cost"], c_inf, 1e-4, what="large-eps cost")
    _close(out["grad"], 2 * a[:, None] * (X - yb[None, :]), 1e-4, what="large-eps grad")


def pin_invariances(orc):
    """Translation leaves f, g, cost unchanged; rotation leaves them unchanged
    and rotates the gradient; shifting the warm start by (c, -c) shifts the
    output by (c, -c); swapping the clouds swaps f and g at convergence."""
    X, Y, a, b = _problem(7, 19, 23, 3)
    eps, it = 0.1, 30
    f, g = orc.sinkhorn(X, Y, a, b, [eps], [it])
    ref = orc.plan_apply(X, Y, a, b, f, g, eps)
    t = np.array([0.7, -1.3, 2.1])
    f2, g2 = orc.sinkhorn(X + t, Y + t, a, b, [eps], [it])
    _close(f2, f, 1e-11, atol=1e-11, what="translation f")
    _close(g2, g, 1e-11, atol=1e-11, what="translation g")
    _close(orc.plan_apply(X + t, Y + t, a, b, f2, g2, eps)["cost"], ref["cost"], 1e-11, what="translation cost")
    th = 0.77
    R = np.array([[np.cos(th), -np.sin(th), 0], [np.sin(th), np.cos(th), 0], [0, 0, 1.0]])
    f3, g3 = orc.sinkhorn(X @ R.T, Y @ R.T, a, b, [eps], [it])
    out3 = orc.plan_apply(X @ R.T, Y @ R.T, a, b, f3, g3, eps)
    _close(out3["cost"], ref["cost"], 1e-11, what="rotation cost")
    _close(out3["grad"], ref["grad"] @ R.T, 1e-10, what="rotation grad")
    # shift invariance through the warm start
    f0, g0 = orc.sinkhorn(X, Y, a, b, [eps], [3])
    c = 0.37
    fa, ga = orc.sinkhorn(X, Y, a, b, [eps], [5], f0=f0, g0=g0)
    fb, gb = orc.sinkhorn(X, Y, a, b, [eps], [5], f0=f0 + c, g0=g0 - c)
    _close(fb, fa + c, 1e-12, atol=1e-12, what="shift f")
    _close(gb, ga - c, 1e-12, atol=1e-12, what="shift g")
    # swap at convergence
    fc, gc = orc.sinkhorn(X, Y, a, b, [eps], [2000])
    fs, gs = orc.sinkhorn(Y, X, b, a, [eps], [2000])
    gs_f, fs_g = _gauge(gs, fs, fc, gc)
    _close(gs_f, fc, 1e-9, atol=1e-9, what="swap f")
    _close(fs_g, gc, 1e-9, atol=1e-9, what="swap g")


def pin_dual_finite_differences(orc):
    """At convergence the gradient equals finite differences of the dual
    objective <a,f> + <b,g> with respect to X (envelope theorem)."""
    X, Y, a, b = _problem(8, 6, 5, 2, scale=0.6)
    eps = 0.3

    def obj(Xp):
        f, g = orc.sinkhorn(Xp, Y, a, b, [eps], [3000])
        return a @ f + b @ g

    f, g = orc.sinkhorn(X, Y, a, b, [eps], [3000])
    grad = orc.plan_apply(X, Y, a, b, f, g, eps)["grad"]
    h = 1e-5
    fd = np.zeros_like(X)
    for i in range(X.shape[0]):
        for k in range(X.shape[1]):
            Xp, Xm = X.copy(), X.copy()
            Xp[i, k] += h
            Xm[i, k] -= h
            fd[i, k] = (obj(Xp) - obj(Xm)) / (2 * h)
    _close(grad, fd, 1e-6, atol=1e-9, what="finite differences of the dual")


def pin_lse_extremes(orc):
    """Half-steps on rows of extreme structure, with closed forms:
    - identical points, a constant g and uniform b: f_i = |x - y|^2 - g exactly;
    - one column far above the rest (its term exceeds the others by e^40):
      f_i = C_ij - g_j - eps log b_j for that column, to fp64 rounding;
    - a spread of 1e4 eps in g: finite, and equal to a log-sum-exp taken
      independently (scipy) on the same scores."""
    rng = _rng(50)
    eps = 0.05
    x, y = rng.normal(size=(1, 3)), rng.normal(size=(1, 3))
    X, Y = np.repeat(x, 6, 0), np.repeat(y, 5, 0)
    c = float(np.sum((x - y) ** 2))
    _close(orc.f_half(X, Y, None, np.full(5, 0.7), eps), np.full(6, c - 0.7), 1e-13, what="all-equal row")
    X, Y = rng.normal(size=(4, 3)), rng.normal(size=(9, 3))
    b = rng.random(9) + 0.1
    b /= b.sum()
    C = ((X[:, None, :] - Y[None, :, :]) ** 2).sum(-1)
    g = np.zeros(9)
    j0 = 4
    # column j0's score beats every other by at least 40 (in units of eps)
    s = -C / eps + np.log(b)[None, :]
    g[j0] = eps * (40.0 + np.max(s - s[:, [j0]]))
    _close(orc.f_half(X, Y, b, g, eps), C[:, j0] - g[j0] - eps * np.log(b[j0]), 1e-14, what="dominant column")
    g = -1e4 * eps * rng.random(9)
    f = orc.f_half(X, Y, b, g, eps)
    assert np.all(np.isfinite(f)), "non-finite f on a wide row"
    ref = -eps * logsumexp((g[None, :] - C) / eps + np.log(b)[None, :], axis=1)
    _close(f, ref, 1e-13, what="wide row")


def pin_marginal_error_shortcut(orc):
    """Row marginal error by definition, sum_i |sum_j P_ij - a_i|, equals the
    shortcut sum_i a_i |exp((f_i - f'_i)/eps) - 1| with f' the next f-half."""
    X, Y, a, b = _problem(9, 33, 21, 3)
    eps = 0.15
    f, g = orc.sinkhorn(X, Y, a, b, [eps], [4])
    fnew = orc.f_half(X, Y, b, g, eps)
    short = np.sum(a * np.abs(np.exp((f - fnew) / eps) - 1.0))
    _close(orc.marginal_err(X, Y, a, b, f, g, eps), short, 1e-10, what="marginal error shortcut")


def pin_maxima_lse_bounds(orc):
    """A maximum lies between the log-sum-exp and the log-sum-exp minus the log
    of the count.  After a g-half, -g_j/eps is the column's log-sum-exp of
    (f_i - C_ij)/eps + log a_i exactly, so -g_j/eps - log n <= Mc_j <= -g_j/eps;
    at convergence the rows obey the same bounds with f and m.  Both bounds
    are attained by a dominant pair at small eps."""
    X, Y, a, b = _problem(49, 13, 11, 2)
    for eps in (0.5, 0.02):
        f, g = orc.sinkhorn(X, Y, a, b, [eps], [4000])
        Mr, Mc = orc.maxima(X, Y, a, b, f, g, eps)
        n, m = len(f), len(g)
        slack = 1e-9 * (1 + np.abs(g / eps).max())
        assert np.all(Mc <= -g / eps + slack) and np.all(Mc >= -g / eps - np.log(n) - slack), "column maxima"
        slack = 1e-9 * (1 + np.abs(f / eps).max())
        assert np.all(Mr <= -f / eps + slack) and np.all(Mr >= -f / eps - np.log(m) - slack), "row maxima"
    # small eps: the maximum carries almost all of the sum
    _close(Mr, -f / eps, 0, atol=np.log(m) * 0.5 + 1e-9, what="row maxima near the LSE at small eps")


def pin_coo_limits(orc):
    """tau = 0 keeps every pair; tau = 1 keeps exactly the row and column
    argmax pairs; tau -> 0 takes the support gradient to the dense gradient,
    with |difference| bounded by 2 (dropped mass) max|x_i - y_j| per row."""
    X, Y, a, b = _problem(10, 25, 18, 3)
    eps = 0.05
    f, g = orc.sinkhorn(X, Y, a, b, [eps], [800])
    full = orc.coo(X, Y, a, b, f, g, eps, 0.0, 3)
    assert len(full["rows"]) == 25 * 18, "tau = 0 must keep every pair"
    C = ((X[:, None, :] - Y[None, :, :]) ** 2).sum(-1)
    s_row = (g[None, :] - C) / eps + np.log(b)[None, :]
    s_col = (f[:, None] - C) / eps + np.log(a)[:, None]
    want = set(zip(range(25), np.argmax(s_row, axis=1))) | set(zip(np.argmax(s_col, axis=0), range(18)))
    one = orc.coo(X, Y, a, b, f, g, eps, 1.0, 3)
    got = set(zip(one["rows"].tolist(), one["cols"].tolist()))
    assert got == {(int(i), int(j)) for i, j in want}, "tau = 1 must keep the argmax pairs only"
    rows_only = orc.coo(X, Y, a, b, f, g, eps, 1.0, 1)
    assert sorted(rows_only["rows"].tolist()) == list(range(25)), "row test keeps one argmax per row"
    dense = orc.plan_apply(X, Y, a, b, f, g, eps)
    gs_full = orc.grad_support(X, Y, full["rows"], full["cols"], full["vals"])
    # on the full support 2 sum_j P_ij (x_i - y_j) = 2 (r_i x_i - sum_j P_ij y_j),
    # which is the dense gradient plus 2 (r_i - a_i) x_i
    want_full = dense["grad"] + 2 * (dense["rowsum"] - a)[:, None] * X
    _close(gs_full, want_full, 1e-10, atol=1e-14, what="full-support gradient")
    for tau in (1e-3, 1e-8):
        sp = orc.coo(X, Y, a, b, f, g, eps, tau, 3)
        gs = orc.grad_support(X, Y, sp["rows"], sp["cols"], sp["vals"])
        kept = np.zeros(25)
        np.add.at(kept, sp["rows"], sp["vals"])
        dropped = dense["rowsum"] - kept
        bound = 2 * dropped * np.sqrt(C.max()) + 1e-12
        assert np.all(np.linalg.norm(gs - gs_full, axis=1) <= bound + 1e-12), "support gradient bound"


def pin_coo_threshold_hand_worked(orc):
    """The thresholded support for 0 < tau < 1 on a 3 x 3 problem worked by hand
    ("CUDA-Optimized APML", Abstract / Innovation: negligible assignments are
    dropped relative to the largest one, in both directions).

    d = 1, eps = 1, x = (0, 1, 3), y = (0, 2, 5), a = (1/2, 1/4, 1/4),
    b = (1/4, 1/4, 1/2), f = (0, 0, 0), g = (0, 1, 0).  C = [[0, 4, 25],
    [1, 1, 16], [9, 1, 4]], and P_ij = a_i b_j exp(f_i + g_j - C_ij).
    Ratios to the row maximum, P_ij / max_j' P_ij':
        row 0: 1, e^-3, e^-24.3      row 1: e^-1, 1, e^-15.3
        row 2: e^-9, 1, e^-3.307     (e^-3 = 0.0498, e^-3.307 = 0.0366)
    Ratios to the column maximum, P_ij / max_i' P_i'j (column j listed down):
        column 0: 1, e^-1/2, e^-9/2  column 1: e^-2.307, 1, 1
        column 2: e^-20.3, e^-12, 1  (e^-1/2 = 0.184, e^-2.307 = 0.0996)
    Each tau below sits between two of these ratios, so every listed pair
    is decided by a margin of 7 % or more, and the boundary pairs (0, 1),
    (2, 2), (0, 1) and (1, 0) fall on either side of it in turn."""
    X = np.array([[0.0], [1.0], [3.0]])
    Y = np.array([[0.0], [2.0], [5.0]])
    a = np.array([0.5, 0.25, 0.25])
    b = np.array([0.25, 0.25, 0.5])
    f = np.zeros(3)
    g = np.array([0.0, 1.0, 0.0])
    P = {(0, 0): 0.125, (0, 1): 0.125 * np.exp(-3.0), (1, 0): 0.0625 * np.exp(-1.0),
         (1, 1): 0.0625, (2, 1): 0.0625, (2, 2): 0.125 * np.exp(-4.0)}
    cases = [
        # (tau, dirs, support)
        (0.03, 1, [(0, 0), (0, 1), (1, 0), (1, 1), (2, 1), (2, 2)]),  # e^-9 < tau < e^-3.307
        (0.04, 1, [(0, 0), (0, 1), (1, 0), (1, 1), (2, 1)]),          # e^-3.307 < tau < e^-3
        (0.06, 1, [(0, 0), (1, 0), (1, 1), (2, 1)]),                  # e^-3 < tau < e^-1
        (0.06, 2, [(0, 0), (0, 1), (1, 0), (1, 1), (2, 1), (2, 2)]),  # e^-9/2 < tau < e^-2.307
        (0.15, 2, [(0, 0), (1, 0), (1, 1), (2, 1), (2, 2)]),          # e^-2.307 < tau < e^-1/2
        (0.20, 2, [(0, 0), (1, 1), (2, 1), (2, 2)]),                  # e^-1/2 < tau < 1
        (0.15, 3, [(0, 0), (1, 0), (1, 1), (2, 1), (2, 2)]),          # union of the two tests
        (0.04, 3, [(0, 0), (0, 1), (1, 0), (1, 1), (2, 1), (2, 2)]),
    ]
    for tau, dirs, want in cases:
        got = orc.coo(X, Y, a, b, f, g, 1.0, tau, dirs)
        pairs = list(zip(got["rows"].tolist(), got["cols"].tolist()))
        assert pairs == want, f"tau = {tau}, dirs = {dirs}: support {pairs}, expected {want}"
        _close(got["vals"], [P[k] for k in want], 1e-14, what=f"stored values, tau = {tau}, dirs = {dirs}")


def pin_anneal_schedule(orc):
    """eps_k = max(1e-3, 0.9^k): 66 geometric stages from 1.0 down to 0.9^65,
    then one clamped stage at 1e-3 (67 in all).  The annealed solve equals a
    replay of its own realised per-stage iteration counts, and reports the
    marginal error of the returned iterate."""
    st = orc.anneal_stages(1.0, 0.9, 1e-3)
    assert len(st) == 67 and st[0] == 1.0 and st[-1] == 1e-3, "annealing stage list"
    _close(st[:-1], 0.9 ** np.arange(66), 1e-13, what="geometric stages")
    X, Y, a, b = _problem(11, 21, 16, 3)
    out = orc.sinkhorn_anneal(X, Y, a, b, 1.0, 0.5, 0.1, 5, 1e-8, 3000)
    eps_list = orc.anneal_stages(1.0, 0.5, 0.1)[: out["stages_done"]]
    f, g = orc.sinkhorn(X, Y, a, b, eps_list, out["stage_iters"])
    assert np.array_equal(f, out["f"]) and np.array_equal(g, out["g"]), "replay differs"
    assert out["converged"] and out["err"] < 1e-8
    _close(orc.marginal_err(X, Y, a, b, f, g, eps_list[-1]), out["err"], 1e-12, what="reported err")
    assert out["iters_done"] == int(np.sum(out["stage_iters"]))



# ---- cosine cost ("FlashSinkhorn", Conclusies: the cost structure also holds
# for the cosine distance after normalisation) ----------------------------------

def pin_cosine_closed_form(orc):
    """n = m = 1, a = b = 1 under the cosine cost: f = C = 2 - 2 cos(x, y),
    g = 0, cost = C and grad = -2 (yhat - (xhat.yhat) xhat) / |x|.  The values
    are worked by hand; the last case is the zero-point convention (a zero
    point normalises to 0: C = 1 against a nonzero point, gradient 0)."""
    r2 = np.sqrt(2.0)
    cases = [
        ([1.0, 0.0, 0.0], [0.0, 2.0, 0.0], 2.0, [0.0, -2.0, 0.0]),
        ([1.0, 1.0, 0.0], [3.0, 0.0, 0.0], 2.0 - r2, [-1.0 / r2, 1.0 / r2, 0.0]),
        ([0.0, 0.0, -2.0], [0.0, 0.0, 5.0], 4.0, [0.0, 0.0, 0.0]),
        ([0.0, 0.0, 0.0], [1.0, 2.0, 2.0], 1.0, [0.0, 0.0, 0.0]),
    ]
    with orc.cost("cosine"):
        for x, y, c, gr in cases:
            X, Y = np.array([x]), np.array([y])
            for eps, it in ((0.05, 1), (0.5, 3)):
                f, g = orc.sinkhorn(X, Y, [1.0], [1.0], [eps], [it])
                _close(f, [c], 1e-12, atol=1e-12, what="cosine f at n=1")
                _close(g, [0.0], 0, atol=1e-12, what="cosine g at n=1")
                out = orc.plan_apply(X, Y, [1.0], [1.0], f, g, eps)
                _close(out["cost"], c, 1e-12, atol=1e-12, what="cosine cost at n=1")
                _close(out["grad"], [gr], 1e-12, atol=1e-12, what="cosine grad at n=1")


def _unit(P):
    return P / np.linalg.norm(P, axis=1, keepdims=True)


def pin_cosine_unit_points(orc):
    """On unit points |x - y|^2 = 2 - 2 x.y: the cosine oracle gives the
    squared-Euclidean oracle's potentials and cost, and its gradient is the
    squared-Euclidean gradient projected off x_i, (I - x_i x_i^T) grad_i."""
    X, Y, a, b = _problem(11, 13, 17, 4)
    X, Y = _unit(X), _unit(Y)
    eps, it = 0.2, 40
    f, g = orc.sinkhorn(X, Y, a, b, [eps], [it])
    ref = orc.plan_apply(X, Y, a, b, f, g, eps)
    with orc.cost("cosine"):
        fc, gc = orc.sinkhorn(X, Y, a, b, [eps], [it])
        out = orc.plan_apply(X, Y, a, b, fc, gc, eps)
    _close(fc, f, 1e-12, atol=1e-12, what="unit points f")
    _close(gc, g, 1e-12, atol=1e-12, what="unit points g")
    _close(out["cost"], ref["cost"], 1e-12, what="unit points cost")
    proj = ref["grad"] - np.sum(ref["grad"] * X, axis=1, keepdims=True) * X
    _close(out["grad"], proj, 1e-11, atol=1e-12, what="unit points grad")


def pin_cosine_scale_invariance(orc):
    """The cosine cost sees directions only: positive per-point scales on X and
    Y leave f, g and the cost unchanged and divide gradient row i by the scale
    of x_i; every gradient row is orthogonal to its point."""
    X, Y, a, b = _problem(12, 11, 9, 3)
    eps, it = 0.1, 30
    rng = _rng(13)
    cx = rng.uniform(0.2, 5.0, size=(X.shape[0], 1))
    cy = rng.uniform(0.2, 5.0, size=(Y.shape[0], 1))
    with orc.cost("cosine"):
        f, g = orc.sinkhorn(X, Y, a, b, [eps], [it])
        out = orc.plan_apply(X, Y, a, b, f, g, eps)
        f2, g2 = orc.sinkhorn(cx * X, cy * Y, a, b, [eps], [it])
        out2 = orc.plan_apply(cx * X, cy * Y, a, b, f2, g2, eps)
    _close(f2, f, 1e-11, atol=1e-12, what="scaled f")
    _close(g2, g, 1e-11, atol=1e-12, what="scaled g")
    _close(out2["cost"], out["cost"], 1e-11, what="scaled cost")
    _close(out2["grad"], out["grad"] / cx, 1e-10, atol=1e-13, what="scaled grad")
    gmax = np.max(np.abs(out["grad"])) * np.max(np.abs(X))
    _close(np.sum(out["grad"] * X, axis=1), np.zeros(X.shape[0]), 0, atol=1e-12 * gmax, what="grad . x")


def pin_cosine_dual_finite_differences(orc):
    """Envelope theorem under the cosine cost: at convergence the gradient
    equals finite differences of <a,f> + <b,g> with respect to X."""
    X, Y, a, b = _problem(14, 6, 5, 3, scale=0.8)
    eps = 0.2
    with orc.cost("cosine"):
        def obj(Xp):
            f, g = orc.sinkhorn(Xp, Y, a, b, [eps], [3000])
            return a @ f + b @ g

        f, g = orc.sinkhorn(X, Y, a, b, [eps], [3000])
        grad = orc.plan_apply(X, Y, a, b, f, g, eps)["grad"]
        h = 1e-5
        fd = np.zeros_like(X)
        for i in range(X.shape[0]):
            for k in range(X.shape[1]):
                Xp, Xm = X.copy(), X.copy()
                Xp[i, k] += h
                Xm[i, k] -= h
                fd[i, k] = (obj(Xp) - obj(Xm)) / (2 * h)
    _close(grad, fd, 1e-6, atol=1e-9, what="cosine finite differences of the dual")


# ---- transport-matrix products ("FlashSinkhorn", Methodologie 3 and its HVP
# paragraph: P V and P^T U streamed without storing P) -------------------------

def pin_transport_closed_form(orc):
    """A 1 x 1 plan worked by hand: x = (0.5, -1), y = (1.5, 1), C = 5; with
    f = 3, g = 1.5, eps = 0.5 the plan is a b exp((3 + 1.5 - 5)/0.5) = a b / e,
    and both products are that scalar times V."""
    x, y = np.array([[0.5, -1.0]]), np.array([[1.5, 1.0]])
    V = np.array([[2.0, -3.0, 0.25]])
    for a, b in (([1.0], [1.0]), ([0.5], [0.25])):
        pv = a[0] * b[0] * np.exp(-1.0)
        for side in (0, 1):
            out = orc.transport(x, y, a, b, [3.0], [1.5], 0.5, V, side=side)
            _close(out, pv * V, 1e-14, what=f"1 x 1 transport side {side}")


def pin_transport_two_point_closed_form(orc):
    """2 x 2 problems at convergence: both transport products equal the
    closed-form plan applied to V (and its transpose to U)."""
    rng = _rng(48)
    for d, eps in ((2, 0.4), (3, 0.9)):
        X, Y = rng.normal(size=(2, d)), rng.normal(size=(2, d))
        a = np.array([0.3, 0.7])
        b = np.array([0.6, 0.4])
        P = two_point_plan(((X[:, None, :] - Y[None, :, :]) ** 2).sum(-1), a, b, eps)
        V, U = rng.normal(size=(2, 3)), rng.normal(size=(2, 5))
        f, g = orc.sinkhorn(X, Y, a, b, [eps], [4000])
        _close(orc.transport(X, Y, a, b, f, g, eps, V, side=0), P @ V, 1e-10, what="2x2 P V")
        _close(orc.transport(X, Y, a, b, f, g, eps, U, side=1), P.T @ U, 1e-10, what="2x2 P^T U")


def pin_transport_marginals(orc):
    """A run ends with a g-half, after which the column marginals are exact:
    P^T 1 = b.  P 1 approaches a as the run converges, and P Y gives the
    gradient 2 (a_i x_i - (P Y)_i) of the plan application."""
    X, Y, a, b = _problem(21, 9, 7, 3)
    eps = 0.3
    f, g = orc.sinkhorn(X, Y, a, b, [eps], [40])
    _close(orc.transport(X, Y, a, b, f, g, eps, np.ones(9), side=1), b, 1e-12, what="P^T 1 = b")
    fc, gc = orc.sinkhorn(X, Y, a, b, [eps], [4000])
    _close(orc.transport(X, Y, a, b, fc, gc, eps, np.ones(7), side=0), a, 1e-9, what="P 1 -> a")
    PY = orc.transport(X, Y, a, b, f, g, eps, Y, side=0)
    ref = orc.plan_apply(X, Y, a, b, f, g, eps)
    _close(2.0 * (a[:, None] * X - PY), ref["grad"], 1e-12, atol=1e-14, what="gradient from P Y")


def pin_transport_adjoint(orc):
    """The two sides are each other's transpose: <U, P V> = <P^T U, V> for any
    U (n x c) and V (m x c), and each is linear in its matrix."""
    X, Y, a, b = _problem(22, 8, 11, 2)
    eps = 0.2
    f, g = orc.sinkhorn(X, Y, a, b, [eps], [25])
    rng = _rng(23)
    U, V, W = rng.normal(size=(8, 3)), rng.normal(size=(11, 3)), rng.normal(size=(11, 3))
    PV = orc.transport(X, Y, a, b, f, g, eps, V, side=0)
    PtU = orc.transport(X, Y, a, b, f, g, eps, U, side=1)
    _close(np.sum(U * PV), np.sum(PtU * V), 1e-12, what="<U, P V> = <P^T U, V>")
    PW = orc.transport(X, Y, a, b, f, g, eps, W, side=0)
    PVW = orc.transport(X, Y, a, b, f, g, eps, 2.0 * V - W, side=0)
    _close(PVW, 2.0 * PV - PW, 1e-12, atol=1e-15, what="linearity")


# ---- Sparse APML on a stored support ("From Theory to Throughput:
# CUDA-Optimized APML", Abstract: adaptive softmax, bidirectional
# symmetrisation and Sinkhorn normalisation run in COO form) ------------------

def _dense_apml(C, a, b, T, iters):
    """The same loss with dense numpy / scipy matrices (every pair stored)."""
    from scipy.special import softmax
    S = -C / T
    P = 0.5 * (softmax(S, axis=1) + softmax(S, axis=0))
    for _ in range(iters):
        P = P * (a / P.sum(axis=1))[:, None]
        P = P * (b / P.sum(axis=0))[None, :]
    return P, float(np.sum(P * C))


def pin_apml_dense_reduction(orc):
    """With every pair stored, sparse APML equals the dense computation
    (row and column softmax by scipy, symmetrisation, normalisations)."""
    X, Y, a, b = _problem(31, 7, 9, 3)
    C = ((X[:, None, :] - Y[None, :, :]) ** 2).sum(-1)
    rows, cols = np.divmod(np.arange(7 * 9), 9)
    for T, iters in ((0.3, 0), (0.3, 5), (2.0, 20)):
        vals, loss = orc.apml_coo(X, Y, a, b, rows, cols, T, iters)
        P, L = _dense_apml(C, a, b, T, iters)
        _close(vals, P.ravel(), 1e-12, what=f"dense reduction P (T={T}, iters={iters})")
        _close(loss, L, 1e-12, what="dense reduction loss")


def pin_apml_permutation_support(orc):
    """One stored entry per row and per column (a permutation): both softmaxes
    are 1, and after the normalisations every value is b of its column, so the
    loss is sum_j b_j C_{sigma(j) j}."""
    X, Y, a, b = _problem(32, 6, 6, 2)
    sigma = np.array([3, 0, 5, 1, 4, 2])
    rows = np.arange(6)
    cols = sigma
    C = ((X[rows] - Y[cols]) ** 2).sum(-1)
    vals, loss = orc.apml_coo(X, Y, a, b, rows, cols, 0.1, 3)
    _close(vals, b[cols], 1e-14, what="permutation values")
    _close(loss, float(np.sum(b[cols] * C)), 1e-13, what="permutation loss")
    vals0, _ = orc.apml_coo(X, Y, a, b, rows, cols, 0.1, 0)
    _close(vals0, np.ones(6), 1e-15, what="softmaxes of single entries")


def pin_apml_marginals_and_large_T(orc):
    """On a thresholded support the last normalisation makes the column sums
    exactly b; with every pair stored and T -> infinity both softmaxes are
    uniform, so the plan is a x b and the loss the a x b average of C."""
    X, Y, a, b = _problem(33, 10, 8, 3)
    f, g = orc.sinkhorn(X, Y, a, b, [0.05], [200])
    sup = orc.coo(X, Y, a, b, f, g, 0.05, 1e-6)
    vals, _ = orc.apml_coo(X, Y, a, b, sup["rows"], sup["cols"], 0.05, 7)
    col = np.zeros(8)
    np.add.at(col, sup["cols"], vals)
    present = np.isin(np.arange(8), sup["cols"])
    _close(col[present], b[present], 1e-13, what="APML column marginals")
    rows, cols = np.divmod(np.arange(10 * 8), 8)
    C = ((X[:, None, :] - Y[None, :, :]) ** 2).sum(-1)
    _, loss = orc.apml_coo(X, Y, a, b, rows, cols, 1e9, 50)
    _close(loss, float(a @ C @ b), 1e-7, what="large-T loss")

def pin_hvp_finite_differences(orc):
    """The Hessian-vector product is the derivative of the converged gradient
    along V: central differences of the gradient, of the potentials (up to
    the constant gauge) and, independently of the gradient formula, second
    differences of the dual objective <a,f> + <b,g> give V^T H V."""
    X, Y, a, b = _problem(41, 7, 6, 3, scale=0.6)
    eps = 0.3
    V = _rng(42).normal(size=X.shape)

    def solve(Xp):
        return orc.sinkhorn(Xp, Y, a, b, [eps], [3000])

    f, g = solve(X)
    hv, fd, gd = orc.hvp(X, Y, a, b, f, g, eps, V, derivs=True)
    h = 1e-5
    fp, gp = solve(X + h * V)
    fm, gm = solve(X - h * V)
    grad = lambda Xp, fq, gq: orc.plan_apply(Xp, Y, a, b, fq, gq, eps)["grad"]
    _close(hv, (grad(X + h * V, fp, gp) - grad(X - h * V, fm, gm)) / (2 * h), 1e-6, what="HVP vs gradient differences")
    dfd, dgd = _gauge((fp - fm) / (2 * h), (gp - gm) / (2 * h), fd, gd)
    _close(dfd, fd, 1e-6, atol=1e-9, what="potential derivative f")
    _close(dgd, gd, 1e-6, atol=1e-9, what="potential derivative g")
    hh = 1e-3
    dual = lambda Xp: (lambda fg: a @ fg[0] + b @ fg[1])(solve(Xp))
    second = (dual(X + hh * V) - 2 * dual(X) + dual(X - hh * V)) / hh ** 2
    _close(np.sum(V * hv), second, 1e-5, what="V^T H V vs second differences of the dual")


def pin_hvp_two_point_closed_form(orc):
    """2 x 2 problems: the gradient 2 sum_j P_ij (x_i - y_j) built from the
    closed-form plan, differentiated along V by central differences, gives
    H V with no Sinkhorn iteration involved."""
    rng = _rng(47)
    for d, eps in ((1, 0.3), (2, 0.5), (3, 1.2)):
        X, Y, V = rng.normal(size=(2, d)), rng.normal(size=(2, d)), rng.normal(size=(2, d))
        a = np.array([0.35, 0.65])
        b = np.array([0.55, 0.45])

        def grad(Xp):
            P = two_point_plan(((Xp[:, None, :] - Y[None, :, :]) ** 2).sum(-1), a, b, eps)
            return 2 * (P[:, :, None] * (Xp[:, None, :] - Y[None, :, :])).sum(1)

        h = 1e-5
        ref = (grad(X + h * V) - grad(X - h * V)) / (2 * h)
        f, g = orc.sinkhorn(X, Y, a, b, [eps], [4000])
        _close(orc.hvp(X, Y, a, b, f, g, eps, V), ref, 1e-7, what=f"2x2 HVP (d = {d})")


def pin_hvp_structure(orc):
    """The Hessian is symmetric (U^T H V = V^T H U); the column marginals stay
    fixed, so sum_i (H V)_i = 2 sum_i a_i v_i at convergence; rotating both
    clouds and V rotates H V; n = m = 1 gives H V = 2 v; as eps -> infinity,
    P -> a x b and H V -> 2 a_i v_i with error O(1 / eps)."""
    X, Y, a, b = _problem(43, 9, 11, 3)
    eps = 0.5
    rng = _rng(44)
    U, V = rng.normal(size=X.shape), rng.normal(size=X.shape)
    f, g = orc.sinkhorn(X, Y, a, b, [eps], [3000])
    hv = orc.hvp(X, Y, a, b, f, g, eps, V)
    hu = orc.hvp(X, Y, a, b, f, g, eps, U)
    _close(np.sum(U * hv), np.sum(V * hu), 1e-10, what="HVP symmetry")
    _close(hv.sum(0), 2 * (a[:, None] * V).sum(0), 1e-10, what="HVP column sum")
    th = 1.1
    R = np.array([[1.0, 0, 0], [0, np.cos(th), -np.sin(th)], [0, np.sin(th), np.cos(th)]])
    f3, g3 = orc.sinkhorn(X @ R.T, Y @ R.T, a, b, [eps], [3000])
    _close(orc.hvp(X @ R.T, Y @ R.T, a, b, f3, g3, eps, V @ R.T), hv @ R.T, 1e-9, what="HVP rotation")
    x, y, v = rng.normal(size=(1, 4)), rng.normal(size=(1, 4)), rng.normal(size=(1, 4))
    f1, g1 = orc.sinkhorn(x, y, [1.0], [1.0], [0.2], [2])
    _close(orc.hvp(x, y, [1.0], [1.0], f1, g1, 0.2, v), 2 * v, 1e-12, what="HVP at n = m = 1")
    big = 1e6
    fb, gb = orc.sinkhorn(X, Y, a, b, [big], [3])
    _close(orc.hvp(X, Y, a, b, fb, gb, big, V), 2 * a[:, None] * V, 1e-4, what="HVP at large eps")


def pin_hvp_transport_decomposition(orc):
    """The page's decomposition: H V assembled from transport-vector and
    transport-matrix products alone (P 1, P^T 1, P Y, P^T V, P^T w, P(g' Y),
    the packed second moments P (y y^T), and conjugate gradients on the
    marginal system, each step one P u and one P^T u) equals the dense
    solve of the same system."""
    X, Y, a, b = _problem(45, 40, 35, 3)
    eps = 0.4
    V = _rng(46).normal(size=X.shape)
    f, g = orc.sinkhorn(X, Y, a, b, [eps], [2000])
    T = lambda W, side: orc.transport(X, Y, a, b, f, g, eps, W, side)
    n, d = X.shape
    m = Y.shape[0]
    r, c = T(np.ones(m), 0), T(np.ones(n), 1)
    PY, PtV = T(Y, 0), T(V, 1)
    w = np.sum(X * V, 1)
    alpha = 2 * r * w - 2 * np.sum(PY * V, 1)
    beta = 2 * T(w, 1) - 2 * np.sum(Y * PtV, 1)
    res = beta - T(alpha / r, 1)
    gd = np.zeros(m)
    z = res / c
    p, rz, r0 = z.copy(), res @ z, np.linalg.norm(res)
    for _ in range(500):  # preconditioned CG on diag(c) - P^T diag(1/r) P
        Sp = c * p - T(T(p, 0) / r, 1)
        step = rz / (p @ Sp)
        gd += step * p
        res -= step * Sp
        if np.linalg.norm(res) <= 1e-12 * r0:
            break
        z = res / c
        rz, rz_old = res @ z, rz
        p = z + (rz / rz_old) * p
    Pg = T(gd, 0)
    fd = (alpha - Pg) / r
    iu = np.triu_indices(d)
    Mp = T((Y[:, :, None] * Y[:, None, :])[:, iu[0], iu[1]], 0)
    M = np.zeros((n, d, d))
    M[:, iu[0], iu[1]] = Mp
    M[:, iu[1], iu[0]] = Mp
    hv = 2 * r[:, None] * V + (2 / eps) * ((fd - 2 * w)[:, None] * (r[:, None] * X - PY) + Pg[:, None] * X
                                           - T(gd[:, None] * Y, 0) + 2 * np.sum(PY * V, 1)[:, None] * X
                                           - 2 * np.einsum("ikl,il->ik", M, V))
    _close(hv, orc.hvp(X, Y, a, b, f, g, eps, V), 1e-9, what="HVP from transport products vs dense solve")


ALL_PINS = [
    pin_closed_form_single_point,
    pin_two_point_closed_form,
    pin_attention_form,
    pin_marginals_and_duality,
    pin_brute_force_assignment,
    pin_sorted_matching_1d,
    pin_large_eps,
    pin_invariances,
    pin_dual_finite_differences,
    pin_lse_extremes,
    pin_marginal_error_shortcut,
    pin_maxima_lse_bounds,
    pin_coo_limits,
    pin_coo_threshold_hand_worked,
    pin_anneal_schedule,
    pin_cosine_closed_form,
    pin_cosine_unit_points,
    pin_cosine_scale_invariance,
    pin_cosine_dual_finite_differences,
    pin_transport_closed_form,
    pin_transport_two_point_closed_form,
    pin_transport_marginals,
    pin_transport_adjoint,
    pin_apml_dense_reduction,
    pin_apml_permutation_support,
    pin_apml_marginals_and_large_T,
    pin_hvp_finite_differences,
    pin_hvp_two_point_closed_form,
    pin_hvp_structure,
    pin_hvp_transport_decomposition,
]
