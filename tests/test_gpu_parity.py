"""GPU path vs the fp64 oracle, element by element, through the C ABI.

Inputs are the seeded workloads of ``sinkhorn_point_cloud_gb300.datagen`` at
sizes the oracle finishes in seconds (several tiles and a ragged tail), plus
the full sizes where the oracle can follow a sample of the outputs.
Tolerance: normwise relative error 1e-4 for potentials (after the gauge fix),
cost and gradient.
"""
import numpy as np
import pytest

from gpu_util import TOL, dev, host, normwise, potentials_error

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def sot():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sinkhorn_point_cloud_gb300 as s
    from sinkhorn_point_cloud_gb300 import build
    build.build()
    return s


def oracle_run(orc, X, Y, a, b, eps, iters, clouds=None):
    idx = range(X.shape[0]) if clouds is None else clouds
    fs, gs, cs, grs = [], [], [], []
    for k in idx:
        f, g = orc.sinkhorn(X[k], Y[k], a[k], b[k], [eps], [iters])
        out = orc.plan_apply(X[k], Y[k], a[k], b[k], f, g, eps)
        fs.append(f); gs.append(g); cs.append(out["cost"]); grs.append(out["grad"])
    return np.stack(fs), np.stack(gs), np.array(cs), np.stack(grs)


def gpu_run(sot, X, Y, a, b, eps, iters, flags=0, uniform=False):
    Xd, Yd = dev(X), dev(Y)
    ad, bd = (None, None) if uniform else (dev(a), dev(b))
    if flags:
        f, g = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=eps, iters_per_stage=iters, max_iters=iters, flags=flags)
    else:
        f, g = sot.sot_potentials(Xd, Yd, ad, bd, eps=eps, iters=iters)
    c, gr, r = sot.sot_plan_apply(Xd, Yd, ad, bd, f, g, eps, rowsum=True, flags=flags & 3)
    torch.cuda.synchronize()
    return host(f), host(g), host(c), host(gr), host(r)


def check(sot, orc, X, Y, a, b, eps, iters, flags=0, uniform=False, clouds=None, tol=TOL):
    f, g, c, gr, _ = gpu_run(sot, X, Y, a, b, eps, iters, flags, uniform)
    sel = list(range(X.shape[0])) if clouds is None else list(clouds)
    fr, gref, cr, grr = oracle_run(orc, X, Y, a, b, eps, iters, sel)
    ef, eg = potentials_error(f[sel], g[sel], fr, gref)
    ec = max(abs(c[k] - cr[i]) / abs(cr[i]) for i, k in enumerate(sel))
    egr = max(normwise(gr[k], grr[i]) for i, k in enumerate(sel))
    msg = f"f {ef:.2e} g {eg:.2e} cost {ec:.2e} grad {egr:.2e}"
    assert ef < tol and eg < tol and ec < tol and egr < tol, msg
    return msg


def test_workload1_full(sot, orc):
    """B=1, n=m=256, d=3 uniform cube, eps=0.01, 100 iterations (the whole workload)."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(1)
    print(check(sot, orc, X, Y, a, b, 0.01, 100, uniform=True))


@pytest.mark.parametrize("n,m", [(512, 512), (700, 555), (1, 300), (257, 1)])
def test_workload2_reduced(sot, orc, n, m):
    """Sphere + rotation clouds, eps=1e-2, 200 iterations, ragged sizes."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=3, n=n, m=m)
    print(check(sot, orc, X, Y, a, b, 1e-2, 200, uniform=True))


def test_workload2_full_size_sampled_clouds(sot, orc):
    """The full batch B=32, n=m=2048 as timed; the oracle follows clouds 0 and 31."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2)
    print(check(sot, orc, X, Y, a, b, 1e-2, 200, uniform=True, clouds=[0, 31]))


@pytest.mark.parametrize("d", [1, 2])
def test_low_dimensions(sot, orc, d):
    rng = np.random.default_rng(40 + d)
    X = rng.random((2, 300, d)).astype(np.float32)
    Y = (rng.random((2, 280, d)) * 0.7 + 0.2).astype(np.float32)
    a = rng.random((2, 300)) + 0.1
    a = (a / a.sum(1, keepdims=True)).astype(np.float32)
    b = rng.random((2, 280)) + 0.1
    b = (b / b.sum(1, keepdims=True)).astype(np.float32)
    print(check(sot, orc, X, Y, a, b, 0.02, 60))


@pytest.mark.parametrize("n,m,d", [(1000, 1100, 64), (300, 257, 5), (129, 70, 17)])
def test_dense_fp32_path(sot, orc, n, m, d):
    """Gaussian clouds with softmax weights (the n=70000, d=64 recipe at reduced size), fp32 path."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=n, m=m, d=d)
    print(check(sot, orc, X, Y, a, b, 0.1, 100, flags=sot.SOT_PREC_FP32))


def test_workload5_reduced_potentials(sot, orc):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(5, B=2, n=1024)
    print(check(sot, orc, X, Y, a, b, 5e-3, 300, uniform=True))


def test_workload5_full_size_sampled_cloud(sot, orc):
    """The full batch B=8, n=m=8192, eps=5e-3, 300 iterations as timed; the
    oracle follows cloud 0 through all 300 iterations (about 4e10 pair
    evaluations: half a minute on 16 cores) and its plan application."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(5)
    print(check(sot, orc, X, Y, a, b, 5e-3, 300, uniform=True, clouds=[0]))


def test_single_point_closed_form(sot):
    """n = m = 1: f = |x - y|^2, g = 0, cost = |x - y|^2, grad = 2 (x - y)."""
    X = np.array([[[0.3, -0.2, 0.9]]], dtype=np.float32)
    Y = np.array([[[-0.4, 0.5, 0.1]]], dtype=np.float32)
    one = np.ones((1, 1), dtype=np.float32)
    f, g, c, gr, r = gpu_run(sot, X, Y, one, one, 0.05, 3)
    C = float(np.sum((X.astype(np.float64) - Y) ** 2))
    assert abs(f[0, 0] + g[0, 0] - C) < 1e-5 * C  # f + g = C holds in every gauge
    assert abs(c[0] - C) < 1e-5 * C
    assert np.allclose(gr[0, 0], 2 * (X[0, 0] - Y[0, 0]), rtol=1e-5, atol=1e-6)
    assert abs(r[0, 0] - 1.0) < 1e-5


def test_large_eps_closed_form(sot):
    """eps -> infinity: cost -> sum a|x|^2 + sum b|y|^2 - 2 xbar_a . ybar_b."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=2000, m=1500, d=64)
    eps = 1e5
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    f, g = sot.sot_potentials(Xd, Yd, ad, bd, eps=eps, iters=3)
    c = host(sot.sot_cost(Xd, Yd, ad, bd, f, g, eps))[0]
    X64, Y64, a64, b64 = X[0].astype(np.float64), Y[0].astype(np.float64), a[0].astype(np.float64), b[0].astype(np.float64)
    c_inf = a64 @ (X64 ** 2).sum(1) + b64 @ (Y64 ** 2).sum(1) - 2 * (a64 @ X64) @ (b64 @ Y64)
    assert abs(c - c_inf) / c_inf < 2e-3, (c, c_inf)


def test_warm_start_shift(sot):
    """A warm start shifted by (c, -c) returns potentials shifted by (c, -c)."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=2, n=300)
    Xd, Yd = dev(X), dev(Y)
    f0, g0 = sot.sot_potentials(Xd, Yd, eps=0.02, iters=5)
    c = 0.25
    f1, g1 = sot.sot_potentials_ex(Xd, Yd, eps=0.02, iters_per_stage=7, max_iters=7, flags=sot.SOT_WARM_START,
                                   f=f0.clone(), g=g0.clone())
    f2, g2 = sot.sot_potentials_ex(Xd, Yd, eps=0.02, iters_per_stage=7, max_iters=7, flags=sot.SOT_WARM_START,
                                   f=f0 + c, g=g0 - c)
    assert normwise(host(f2) - c, host(f1)) < 1e-5
    assert normwise(host(g2) + c, host(g1)) < 1e-5


@pytest.mark.parametrize("shift", [+60.0, -60.0])
def test_far_warm_start_takes_the_slow_paths(sot, orc, shift):
    """Potentials far from the solution force the tile re-stabilisation
    (overflow side) and the full-row recompute (underflow side); the answer
    must still match the oracle started from the same point."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=1, n=600, m=500)
    eps = 0.01
    f0 = np.full((1, 600), shift, dtype=np.float32)
    g0 = np.zeros((1, 500), dtype=np.float32)
    Xd, Yd = dev(X), dev(Y)
    f, g = sot.sot_potentials_ex(Xd, Yd, eps=eps, iters_per_stage=20, max_iters=20, flags=sot.SOT_WARM_START,
                                 f=dev(f0), g=dev(g0))
    fr, gr = orc.sinkhorn(X[0], Y[0], None, None, [eps], [20], f0=f0[0], g0=g0[0])
    ef, eg = potentials_error(host(f), host(g), fr[None], gr[None])
    assert ef < TOL and eg < TOL, (ef, eg)


def test_bitwise_reproducible(sot):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=4, n=1500)
    Xd, Yd = dev(X), dev(Y)
    f1, g1 = sot.sot_potentials(Xd, Yd, eps=0.01, iters=20)
    f2, g2 = sot.sot_potentials(Xd, Yd, eps=0.01, iters=20)
    assert torch.equal(f1, f2) and torch.equal(g1, g2)


def test_dense_fp32_path_d256(sot, orc):
    """d = 256, the largest dimension whose rows stay staged whole."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=200, m=170, d=256)
    assert sot.sot_select_path(256, sot.SOT_PREC_FP32) == 1
    print(check(sot, orc, X, Y, a, b, 2.0, 60, flags=sot.SOT_PREC_FP32))


@pytest.mark.parametrize("d,n,m,B", [(512, 200, 170, 1), (1000, 130, 111, 2), (1024, 97, 140, 1)])
def test_dense_fp32_path_wide_d(sot, orc, d, n, m, B):
    """d = 512, a ragged 1000 and the largest, 1024 ("FlashSinkhorn",
    Experimentele Resultaten: d up to 1024) on the fp32 path: the coordinates
    stream in slices of 256 and the plan application takes the gradient in
    256-coordinate slices, with the significant pairs' weights exact.  eps
    grows with d, as the costs do."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=B, n=n, m=m, d=d)
    assert sot.sot_select_path(d, sot.SOT_PREC_FP32) == 1
    print(check(sot, orc, X, Y, a, b, d / 128.0, 60, flags=sot.SOT_PREC_FP32))
