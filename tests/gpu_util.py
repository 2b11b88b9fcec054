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
    relative to the common scale max(|f_ref|_inf, |g_ref|_inf): the two
    potentials share one gauge and one scale (f_i + g_j ~ C_ij), and one of
    them can sit near zero (e.g. a single target point has g = 0)."""
    ef, eg = 0.0, 0.0
    for k in range(f.shape[0]):
        fk, gk = gauge_fixed(f[k], g[k], fr[k], gr[k])
        scale = max(np.max(np.abs(fr[k])), np.max(np.abs(gr[k])), 1e-300)
        ef = max(ef, float(np.max(np.abs(fk - fr[k])) / scale))
        eg = max(eg, float(np.max(np.abs(gk - gr[k])) / scale))
    return ef, eg
