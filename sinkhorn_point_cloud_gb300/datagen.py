"""Seeded synthetic point clouds for the five workloads of this library.

This module only draws random inputs; it holds none of the transport
arithmetic, so both the CUDA path and the fp64 CPU oracle can consume the same
arrays.  Every array is drawn in float64 from ``numpy.random.Generator(PCG64)``
and cast once to float32; those float32 arrays are the ground truth that both
sides read.

The pages measure on ShapeNet / MM-Fi point clouds ("From Theory to Throughput:
CUDA-Optimized APML", Abstract) and on synthetic EOT problems up to n = 70,000
("FlashSinkhorn", Probleemstelling; Experimentele Resultaten).  None of those
datasets is available, so the distributions below stand in for them:

* ``uniform01``  X, Y i.i.d. uniform in [0,1]^d, uniform weights.
* ``sphere_rot`` X = unit-sphere points + N(0, 0.01^2); Y = X R^T + N(0, 0.01^2)
  with R a Haar-random rotation in SO(3) per cloud; uniform weights.
* ``gmm``        X and Y independent 8-component Gaussian mixtures in 3-D, means
  U[-1,1]^3 (drawn separately for X and Y), std 0.05, equal component weights;
  uniform weights.
* ``gauss``      X ~ N(0, I_d), Y ~ N(mu, I_d) with mu ~ N(0, 0.25 I_d) per
  problem; a, b = softmax of independent N(0,1) logits.

Seeds: cloud ``k`` of workload ``w`` uses ``seed = 20260000 + 100*w + k`` unless
a ``seed_base`` is given.
"""
from __future__ import annotations

import numpy as np

# Workload table: the five configurations (sizes, eps, schedule, data recipe).
WORKLOADS = {
    1: dict(name="uniform01_n256_d3", B=1, n=256, m=256, d=3, kind="uniform01",
            eps=0.01, iters=100),
    2: dict(name="sphere_rot_B32_n2048_d3", B=32, n=2048, m=2048, d=3, kind="sphere_rot",
            eps=1e-2, iters=200),
    3: dict(name="gmm8_B4_n16384_d3_annealed", B=4, n=16384, m=16384, d=3, kind="gmm",
            eps=1e-3, eps_init=1.0, eps_factor=0.9, iters_per_stage=20, tol=1e-4,
            max_iters=5000),
    4: dict(name="gauss_n70000_d64", B=1, n=70000, m=70000, d=64, kind="gauss",
            eps=0.1, iters=100),
    5: dict(name="sphere_rot_B8_n8192_d3_coo", B=8, n=8192, m=8192, d=3, kind="sphere_rot",
            eps=5e-3, iters=300, tau=1e-8),
}


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def haar_so3(rng: np.random.Generator) -> np.ndarray:
    """Haar-distributed rotation: QR of a Gaussian matrix with the sign fix, det = +1."""
    z = rng.standard_normal((3, 3))
    q, r = np.linalg.qr(z)
    q = q * np.sign(np.diag(r))[None, :]
    if np.linalg.det(q) < 0:
        q[:, 0] = -q[:, 0]
    return q


def _unit_sphere(rng, n):
    v = rng.standard_normal((n, 3))
    return v / np.linalg.norm(v, axis=1, keepdims=True)


def _gmm(rng, n, k=8, sigma=0.05):
    means = rng.uniform(-1.0, 1.0, size=(k, 3))
    comp = rng.integers(0, k, size=n)
    return means[comp] + sigma * rng.standard_normal((n, 3))


def _softmax(z):
    z = z - z.max()
    e = np.exp(z)
    return e / e.sum()


def make_cloud(kind: str, n: int, m: int, d: int, seed: int):
    """One problem (X[n,d], Y[m,d], a[n], b[m]) as float32 arrays."""
    rng = _rng(seed)
    if kind == "uniform01":
        X = rng.uniform(0.0, 1.0, size=(n, d))
        Y = rng.uniform(0.0, 1.0, size=(m, d))
        a = np.full(n, 1.0 / n)
        b = np.full(m, 1.0 / m)
    elif kind == "sphere_rot":
        if d != 3:
            raise ValueError("sphere_rot is a 3-D recipe")
        X = _unit_sphere(rng, n) + 0.01 * rng.standard_normal((n, 3))
        R = haar_so3(rng)
        if m <= n:
            base = X[:m]
        else:  # more targets than sources: extra targets are fresh sphere points
            base = np.concatenate([X, _unit_sphere(rng, m - n)], axis=0)
        Y = base @ R.T + 0.01 * rng.standard_normal((m, 3))
        a = np.full(n, 1.0 / n)
        b = np.full(m, 1.0 / m)
    elif kind == "gmm":
        if d != 3:
            raise ValueError("gmm is a 3-D recipe")
        X = _gmm(rng, n)
        Y = _gmm(rng, m)
        a = np.full(n, 1.0 / n)
        b = np.full(m, 1.0 / m)
    elif kind == "gauss":
        mu = 0.5 * rng.standard_normal(d)
        X = rng.standard_normal((n, d))
        Y = mu[None, :] + rng.standard_normal((m, d))
        a = _softmax(rng.standard_normal(n))
        b = _softmax(rng.standard_normal(m))
    else:
        raise ValueError(f"unknown data kind {kind!r}")
    f32 = lambda v: np.ascontiguousarray(v, dtype=np.float32)
    return f32(X), f32(Y), f32(a), f32(b)


def make_batch(workload: int, B: int | None = None, n: int | None = None,
               m: int | None = None, d: int | None = None, seed_base: int | None = None,
               clouds=None):
    """Batch of problems of a workload, optionally resized.

    Returns X[B,n,d], Y[B,m,d], a[B,n], b[B,m] (float32, C-contiguous).  ``clouds``
    selects cloud indices (default ``range(B)``) so a subset of a large batch
    reproduces exactly the same clouds as the full batch.
    """
    w = WORKLOADS[workload]
    B = w["B"] if B is None else B
    if m is None:
        m = w["m"] if n is None else n
    n = w["n"] if n is None else n
    d = w["d"] if d is None else d
    base = 20260000 + 100 * workload if seed_base is None else seed_base
    idx = list(range(B)) if clouds is None else list(clouds)
    parts = [make_cloud(w["kind"], n, m, d, base + k) for k in idx]
    X = np.stack([p[0] for p in parts])
    Y = np.stack([p[1] for p in parts])
    a = np.stack([p[2] for p in parts])
    b = np.stack([p[3] for p in parts])
    return X, Y, a, b
