"""Helpers shared by the GPU parity tests (comparison metrics, device copies)."""
from __future__ import annotations

import numpy as np

# Tolerances.  North-star gates: potentials, cost and gradient within a
# normwise relative error of 1e-4 for the fp32 contraction (also used for the
# fp16 x3 tensor-core products, whose error is below fp32's).
TOL = 1e-4


def dev(x):
    import torch
    return None if x is None else torch.from_numpy(np.ascontiguousarray(x)).cuda()


def host(t):
    return t.detach().cpu().numpy().astype(np.float64)


def normwise(got, ref):
    """max|got - ref| / max|ref| (per whole array)."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.max(np.abs(ref))
    return float(np.max(np.abs(got - ref)) / (den if den > 0 else 1.0))


def gauge_fixed(f, g, fr, gr):
    """Remove the common constant mode (f + c, g - c) before comparing:
    c* = (mean(f - fr) - mean(g - gr)) / 2."""
    c = 0.5 * (np.mean(f - fr) - np.mean(g - gr))
    return f - c, g + c


def potentials_error(f, g, fr, gr):
    """Errors of f and g after the gauge fix (per cloud, max over clouds), each
    relative to the common scale max(|f_ref|_inf, |g_ref|_inf).

    f and g are defined together, up to the gauge (f + c, g - c), and every
    output depends on them through f_i + g_j, which is of the size of C_ij; so
    both are measured against the scale they share.  Measured against its
    own norm instead, a potential that sits near zero (a single target point
    has g = 0 exactly) would turn rounding noise into an unbounded relative
    error.  The per-vector errors |df|_inf / |f_ref|_inf and
    |dg|_inf / |g_ref|_inf are printed beside the joint ones, so a failing
    test shows both."""
    ef, eg, of, og = 0.0, 0.0, 0.0, 0.0
    for k in range(f.shape[0]):
        fk, gk = gauge_fixed(f[k], g[k], fr[k], gr[k])
        nf, ng = np.max(np.abs(fr[k])), np.max(np.abs(gr[k]))
        scale = max(nf, ng, 1e-300)
        df, dg = float(np.max(np.abs(fk - fr[k]))), float(np.max(np.abs(gk - gr[k])))
        ef, eg = max(ef, df / scale), max(eg, dg / scale)
        of, og = max(of, df / max(nf, 1e-300)), max(og, dg / max(ng, 1e-300))
    print(f"potentials (gauge-fixed): joint scale f {ef:.2e} g {eg:.2e}; per-vector f {of:.2e} g {og:.2e}")
    return ef, eg
