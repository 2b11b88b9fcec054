"""Transport-matrix products P V and P^T U ("FlashSinkhorn", Methodologie 3
and its HVP paragraph) through the C ABI vs the fp64 oracle, element by
element, from the GPU's own potentials.

Cases: the sphere + rotation recipe (d = 3) at two column counts and both
sides, a d = 8 Gaussian problem, the n = 70000 recipe (d = 64) at a ragged
reduced size with 64 columns, the cosine cost, and properties that hold at any
size: exact column marginals after the g-half, adjointness on the device.
Tolerance: normwise 1e-4."""
import numpy as np
import pytest

from gpu_util import TOL, dev, host, normwise

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


def potentials(sot, X, Y, a, b, eps, iters, flags=0):
    f, g = sot.sot_potentials_ex(dev(X), dev(Y), dev(a), dev(b), eps=eps, iters_per_stage=iters, max_iters=iters,
                                 flags=flags)
    torch.cuda.synchronize()
    return f, g


def check(sot, orc, X, Y, a, b, eps, iters, c, seed, flags=0, cost="sqeuclidean"):
    f, g = potentials(sot, X, Y, a, b, eps, iters, flags)
    rng = np.random.default_rng(seed)
    B, n, m = X.shape[0], X.shape[1], Y.shape[1]
    errs = []
    for side in (0, 1):
        V = rng.normal(size=(B, m if side == 0 else n, c)).astype(np.float32)
        out = host(sot.sot_transport_apply(dev(X), dev(Y), dev(a), dev(b), f, g, eps, dev(V), side=side,
                                           flags=flags))
        fh, gh = host(f), host(g)
        with orc.cost(cost):
            ref = np.stack([orc.transport(X[k], Y[k], a[k], b[k], fh[k], gh[k], eps, V[k], side=side)
                            for k in range(B)])
        errs.append(max(normwise(out[k], ref[k]) for k in range(B)))
    print(f"P V {errs[0]:.2e}  P^T U {errs[1]:.2e}")
    assert max(errs) < TOL, errs


@pytest.mark.parametrize("c", [1, 5])
def test_transport_point_clouds(sot, orc, c):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=2, n=300, m=257)
    check(sot, orc, X, Y, a, b, 0.01, 100, c, 80 + c)


def test_transport_d8(sot, orc):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=200, m=190, d=8)
    check(sot, orc, X, Y, a, b, 0.1, 60, 16, 90)


def test_transport_d64_reduced(sot, orc):
    """The n = 70000, d = 64 recipe at 600 x 520 (several row tiles, ragged
    column tiles), 64 columns (the largest c)."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=600, m=520)
    check(sot, orc, X, Y, a, b, 0.1, 60, 64, 91)


def test_transport_cosine(sot, orc):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=260, m=300, d=16)
    check(sot, orc, X, Y, a, b, 0.05, 40, 3, 92, flags=sot.SOT_COST_COSINE, cost="cosine")


def test_transport_marginals_and_adjoint(sot):
    """After the g-half the column sums of P are b (to the fp32 rounding of g),
    P 1 is the row marginal, and <U, P V> = <P^T U, V>."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=3, n=700, m=650)
    eps = 0.01
    f, g = potentials(sot, X, Y, a, b, eps, 200)
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    col = host(sot.sot_transport_apply(Xd, Yd, ad, bd, f, g, eps, torch.ones(3, 700, device="cuda"), side=1))
    assert normwise(col, b) < 1e-4, normwise(col, b)
    row = host(sot.sot_transport_apply(Xd, Yd, ad, bd, f, g, eps, torch.ones(3, 650, device="cuda"), side=0))
    _, _, rs = sot.sot_plan_apply(Xd, Yd, ad, bd, f, g, eps, cost=False, grad=False, rowsum=True)
    assert normwise(row, host(rs)) < 1e-4
    rng = np.random.default_rng(93)
    U = rng.normal(size=(3, 700, 4)).astype(np.float32)
    V = rng.normal(size=(3, 650, 4)).astype(np.float32)
    PV = host(sot.sot_transport_apply(Xd, Yd, ad, bd, f, g, eps, dev(V), side=0))
    PtU = host(sot.sot_transport_apply(Xd, Yd, ad, bd, f, g, eps, dev(U), side=1))
    lhs, rhs = np.sum(U * PV, axis=(1, 2)), np.sum(PtU * V, axis=(1, 2))
    scale = np.sum(np.abs(U) * np.abs(PV), axis=(1, 2))
    assert float(np.max(np.abs(lhs - rhs) / scale)) < 1e-5


@pytest.mark.parametrize("w,n,m,d,eps,cosine", [
    (2, 300, 257, 3, 0.01, False),    # point clouds
    (4, 200, 190, 8, 0.1, False),     # d = 8
    (4, 300, 280, 100, 0.5, False),   # d = 100: two products of 64 + 36 coordinates
    (4, 260, 300, 16, 0.05, True),    # cosine cost
])
def test_grad_y(sot, orc, w, n, m, d, eps, cosine):
    """grad_y = 2 (b_j y_j - sum_i P_ij x_i) vs the oracle's gradient of the
    swapped problem (Y, X, b, a, g, f), which is the same quantity."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(w, B=2, n=n, m=m, d=d)
    fl = sot.SOT_COST_COSINE if cosine else 0
    f, g = potentials(sot, X, Y, a, b, eps, 60, fl)
    gy = host(sot.sot_grad_y(dev(X), dev(Y), dev(a), dev(b), f, g, eps, flags=fl))
    fh, gh = host(f), host(g)
    with orc.cost("cosine" if cosine else "sqeuclidean"):
        ref = [orc.plan_apply(Y[k], X[k], b[k], a[k], gh[k], fh[k], eps)["grad"] for k in range(2)]
    err = max(normwise(gy[k], ref[k]) for k in range(2))
    print(f"grad_y {err:.2e}")
    assert err < TOL, err


def test_transport_full_size_sampled_rows(sot, orc):
    """The n = m = 70000, d = 64 recipe at full size (the bench's launch
    configuration: 3 column chunks), potentials after 3 iterations; P V with
    4 columns against the oracle on 12 sampled rows (a row of P V needs only
    its own point, potential and weight, and every column)."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4)
    f, g = potentials(sot, X, Y, a, b, 0.1, 3)
    rng = np.random.default_rng(94)
    V = rng.normal(size=(1, 70000, 4)).astype(np.float32)
    out = host(sot.sot_transport_apply(dev(X), dev(Y), dev(a), dev(b), f, g, 0.1, dev(V), side=0))
    rows = np.sort(rng.choice(70000, size=12, replace=False))
    fh, gh = host(f), host(g)
    ref = orc.transport(X[0][rows], Y[0], a[0][rows], b[0], fh[0][rows], gh[0], 0.1, V[0], side=0)
    err = normwise(out[0][rows], ref)
    print(f"full size, sampled rows: {err:.2e}")
    assert err < TOL, err


def test_transport_largest_d_and_c(sot, orc):
    """d = 256 and c = 64, the largest the call takes (175 KB of shared memory per CTA)."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=150, m=140, d=256)
    check(sot, orc, X, Y, a, b, 2.0, 30, 64, 95)


def test_grad_y_largest_d(sot, orc):
    """d = 256: four transport products of 64 coordinates."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=120, m=110, d=256)
    f, g = potentials(sot, X, Y, a, b, 2.0, 30)
    gy = host(sot.sot_grad_y(dev(X), dev(Y), dev(a), dev(b), f, g, 2.0))
    ref = orc.plan_apply(Y[0], X[0], b[0], a[0], host(g)[0], host(f)[0], 2.0)["grad"]
    err = normwise(gy[0], ref)
    print(f"grad_y d=256 {err:.2e}")
    assert err < TOL, err
