"""Hessian-vector product on the device (sot_hvp) against the oracle's dense solve.

"FlashSinkhorn", Methodologie 3, HVP paragraph: the product is streamed as
transport-vector and transport-matrix products.  Both sides take the same fp32
potentials (the oracle's converged ones, rounded).  The tolerance is the fp32
floor of the route (design notes, reading 15): conjugate gradients to a 1e-5
relative residual on products whose own error is ~1e-6, and a row-centred
assembly; simulated in fp32 at 1.5e-5 to 5e-5.  The test holds it to 1e-4.
"""
import numpy as np
import pytest

from gpu_util import dev, host, normwise

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

TOL = 1e-4


@pytest.fixture(scope="module")
def sot():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sinkhorn_point_cloud_gb300 as s
    from sinkhorn_point_cloud_gb300 import build
    build.build()
    return s


def _potentials(orc, X, Y, a, b, eps, iters):
    fs, gs = [], []
    for k in range(X.shape[0]):
        f, g = orc.sinkhorn(X[k], Y[k], None if a is None else a[k], None if b is None else b[k], [eps], [iters])
        fs.append(f.astype(np.float32))
        gs.append(g.astype(np.float32))
    return np.stack(fs), np.stack(gs)


def _compare(sot, orc, X, Y, a, b, eps, iters, seed):
    f, g = _potentials(orc, X, Y, a, b, eps, iters)
    V = np.random.default_rng(seed).normal(size=X.shape).astype(np.float32)
    hv = host(sot.sot_hvp(dev(X), dev(Y), dev(a), dev(b), dev(f), dev(g), eps, dev(V)))
    worst = 0.0
    for k in range(X.shape[0]):
        ref = orc.hvp(X[k], Y[k], None if a is None else a[k], None if b is None else b[k], f[k], g[k], eps, V[k])
        worst = max(worst, normwise(hv[k], ref))
    print(f"H V: {worst:.2e}")
    return worst


@pytest.mark.parametrize("n,m", [(256, 256), (301, 257)])
def test_hvp_uniform_cube(sot, orc, n, m):
    """The 256-point uniform recipe (d = 3) at eps = 0.02, and a ragged size."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(1, B=1, n=n, m=m)
    assert _compare(sot, orc, X, Y, None, None, 0.02, 300, 11) < TOL


def test_hvp_sphere_batch(sot, orc):
    """Three clouds of the sphere recipe in one call, each against its own solve."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=3, n=300, m=280)
    assert _compare(sot, orc, X, Y, None, None, 0.02, 400, 13) < TOL


def test_hvp_weighted_d8(sot, orc):
    """Non-uniform weights, d = 8 (the Gaussian recipe cut to 8 dimensions)."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=200, m=190, d=8)
    assert _compare(sot, orc, X, Y, a, b, 0.5, 400, 12) < TOL


def test_hvp_structure(sot, orc):
    """V = 0 gives exactly 0; U^T H V = V^T H U; a common translation of both
    clouds leaves H V unchanged; sum_i (H V)_i = 2 sum_i a_i v_i (the plan's
    column sums are fixed, so moving X moves no mass between columns)."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(1, B=1, n=150, m=140)
    eps = 0.05
    f, g = _potentials(orc, X, Y, None, None, eps, 400)
    fd, gd = dev(f), dev(g)
    zero = host(sot.sot_hvp(dev(X), dev(Y), None, None, fd, gd, eps, dev(np.zeros_like(X))))
    assert np.all(zero == 0.0)
    rng = np.random.default_rng(14)
    U = rng.normal(size=X.shape).astype(np.float32)
    V = rng.normal(size=X.shape).astype(np.float32)
    hu = host(sot.sot_hvp(dev(X), dev(Y), None, None, fd, gd, eps, dev(U)))
    hv = host(sot.sot_hvp(dev(X), dev(Y), None, None, fd, gd, eps, dev(V)))
    lhs, rhs = float(np.sum(U * hv)), float(np.sum(V * hu))
    assert abs(lhs - rhs) <= TOL * max(abs(lhs), abs(rhs)), (lhs, rhs)
    t = np.array([3.0, -2.0, 5.0], np.float32)
    ht = host(sot.sot_hvp(dev(X + t), dev(Y + t), None, None, fd, gd, eps, dev(V)))
    assert normwise(ht, hv) < TOL
    colsum = hv[0].sum(0)
    want = 2.0 * V[0].astype(np.float64).sum(0) / X.shape[1]
    assert np.max(np.abs(colsum - want)) <= TOL * np.max(np.abs(hv)) * X.shape[1] ** 0.5, (colsum, want)


def test_hvp_rejects_bad_arguments(sot):
    X = torch.zeros(1, 8, 10, device="cuda")
    f = torch.zeros(1, 8, device="cuda")
    with pytest.raises(sot.SotError) as ei:
        sot.sot_hvp(X, X, None, None, f, f, 0.1, X)
    assert ei.value.status == sot.SOT_ERR_UNSUPPORTED
    X3 = torch.zeros(1, 8, 3, device="cuda")
    with pytest.raises(sot.SotError) as ei:
        sot.sot_hvp(X3, X3, None, None, f, f, 0.1, X3, cg_iters=0)
    assert ei.value.status == sot.SOT_ERR_INVALID_ARG
