"""Cosine cost (SOT_COST_COSINE; "FlashSinkhorn", Conclusies: the structure
holds for the cosine distance after normalisation) on the point, fp32 and
tensor-core paths vs the fp64 oracle under the cosine cost, element by element.

The clouds of the sphere and Gaussian recipes get per-point scales spread
over [0.2, 5] (the cost must not see them) and, on the point path, one zero
point (it normalises to the zero vector).  Tolerance: normwise 1e-4, as for
the squared-Euclidean cost."""
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


def scaled(X, Y, seed, zero_point=False):
    rng = np.random.default_rng(seed)
    cx = rng.uniform(0.2, 5.0, size=X.shape[:2] + (1,))
    cy = rng.uniform(0.2, 5.0, size=Y.shape[:2] + (1,))
    if zero_point:
        cx[0, 3] = 0.0
    return (X * cx).astype(np.float32), (Y * cy).astype(np.float32)


def gpu_cosine(sot, X, Y, a, b, eps, iters, prec=0):
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    fl = sot.SOT_COST_COSINE | prec
    f, g = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=eps, iters_per_stage=iters, max_iters=iters, flags=fl)
    c, gr, r = sot.sot_plan_apply(Xd, Yd, ad, bd, f, g, eps, rowsum=True, flags=fl)
    torch.cuda.synchronize()
    return host(f), host(g), host(c), host(gr)


def oracle_cosine(orc, X, Y, a, b, eps, iters):
    fs, gs, cs, grs = [], [], [], []
    with orc.cost("cosine"):
        for k in range(X.shape[0]):
            f, g = orc.sinkhorn(X[k], Y[k], a[k], b[k], [eps], [iters])
            out = orc.plan_apply(X[k], Y[k], a[k], b[k], f, g, eps)
            fs.append(f); gs.append(g); cs.append(out["cost"]); grs.append(out["grad"])
    return np.stack(fs), np.stack(gs), np.array(cs), np.stack(grs)


def check(sot, orc, X, Y, a, b, eps, iters, prec=0):
    f, g, c, gr = gpu_cosine(sot, X, Y, a, b, eps, iters, prec)
    fr, gref, cr, grr = oracle_cosine(orc, X, Y, a, b, eps, iters)
    ef, eg = potentials_error(f, g, fr, gref)
    ec = float(np.max(np.abs(c - cr) / np.abs(cr)))
    egr = max(normwise(gr[k], grr[k]) for k in range(X.shape[0]))
    msg = f"f {ef:.2e} g {eg:.2e} cost {ec:.2e} grad {egr:.2e}"
    print(msg)
    assert ef < TOL and eg < TOL and ec < TOL and egr < TOL, msg
    return f, g, c, gr


def test_cosine_point_path(sot, orc):
    """d = 3 (point path): sphere + rotation clouds with spread scales and a zero point."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=2, n=300, m=257)
    X, Y = scaled(X, Y, 71, zero_point=True)
    assert sot.sot_select_path(3, 0) == 0
    check(sot, orc, X, Y, a, b, 0.05, 60)


def test_cosine_fp32_path(sot, orc):
    """d = 8 (fp32 path, d not a multiple of 16): Gaussian clouds, softmax weights."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=200, m=190, d=8)
    X, Y = scaled(X, Y, 72)
    check(sot, orc, X, Y, a, b, 0.05, 80)


def test_cosine_tensor_path(sot, orc):
    """d = 64 (tensor-core path, screened warm half-steps): the n = 70000 recipe
    at a ragged reduced size spanning several row blocks and column tiles."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=600, m=520)
    X, Y = scaled(X, Y, 73)
    assert sot.sot_select_path(64, 0) == 2
    check(sot, orc, X, Y, a, b, 0.02, 60)


def test_cosine_scale_invariance_on_device(sot):
    """Potentials and cost do not see per-point scales; gradient rows divide by
    the scale of their point and are orthogonal to it."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=2, n=400, m=380)
    f1, g1, c1, gr1 = gpu_cosine(sot, X, Y, a, b, 0.05, 40)
    rng = np.random.default_rng(74)
    cx = rng.uniform(0.2, 5.0, size=X.shape[:2] + (1,)).astype(np.float32)
    f2, g2, c2, gr2 = gpu_cosine(sot, (X * cx).astype(np.float32), Y, a, b, 0.05, 40)
    ef, eg = potentials_error(f2, g2, f1, g1)
    assert ef < 2e-6 and eg < 2e-6, (ef, eg)
    assert float(np.max(np.abs(c2 - c1) / np.abs(c1))) < 2e-6
    assert normwise(gr2 * cx, gr1) < 1e-5
    dots = np.abs(np.sum(gr1 * X, axis=2)) / (np.max(np.abs(gr1)) * np.max(np.abs(X)))
    assert float(np.max(dots)) < 1e-5


def test_cosine_equals_squared_euclidean_on_unit_points(sot):
    """On unit points the cosine run and the plain run give the same potentials
    and cost (|x - y|^2 = 2 - 2 x.y there)."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=300, m=310, d=16)
    X = (X / np.linalg.norm(X, axis=2, keepdims=True)).astype(np.float32)
    Y = (Y / np.linalg.norm(Y, axis=2, keepdims=True)).astype(np.float32)
    f1, g1, c1, _ = gpu_cosine(sot, X, Y, a, b, 0.05, 40)
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    f, g = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=0.05, iters_per_stage=40, max_iters=40, flags=0)
    c, _, _ = sot.sot_plan_apply(Xd, Yd, ad, bd, f, g, 0.05, grad=False, rowsum=False)
    torch.cuda.synchronize()
    ef, eg = potentials_error(f1, g1, host(f), host(g))
    assert ef < 1e-5 and eg < 1e-5, (ef, eg)
    assert abs(c1[0] - host(c)[0]) / abs(host(c)[0]) < 1e-5
