"""Sparse APML on a stored support ("From Theory to Throughput: CUDA-Optimized
APML", Abstract and Innovation) through the C ABI vs the fp64 oracle, entry by
entry: supports from sot_plan_coo on the sphere + rotation recipe (d = 3) and
a Gaussian d = 8 problem, every pair stored (tau = 0), 0 and several
normalisations; invalid supports are rejected.  Tolerance: normwise 1e-4."""
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


def support(sot, X, Y, a, b, eps, iters, tau, weighted):
    Xd, Yd = dev(X), dev(Y)
    ad, bd = (dev(a), dev(b)) if weighted else (None, None)
    f, g = sot.sot_potentials(Xd, Yd, ad, bd, eps=eps, iters=iters)
    coo = sot.sot_plan_coo(Xd, Yd, ad, bd, f, g, eps, threshold=tau, dirs=3)
    torch.cuda.synchronize()
    return Xd, Yd, ad, bd, coo


def check(sot, orc, X, Y, a, b, eps, iters, tau, T, norm_iters, weighted=False):
    Xd, Yd, ad, bd, coo = support(sot, X, Y, a, b, eps, iters, tau, weighted)
    vals, loss, grad = sot.sot_apml_coo(Xd, Yd, ad, bd, coo, T, norm_iters)
    torch.cuda.synchronize()
    vals, loss, grad = host(vals), host(loss), host(grad)
    rows, cols, off = host(coo["rows"]).astype(np.int64), host(coo["cols"]).astype(np.int64), \
        host(coo["batch_offsets"]).astype(np.int64)
    ev = el = eg = 0.0
    for k in range(X.shape[0]):
        s0, s1 = off[k], off[k + 1]
        aw = a[k] if weighted else None
        bw = b[k] if weighted else None
        rv, rl = orc.apml_coo(X[k], Y[k], aw, bw, rows[s0:s1], cols[s0:s1], T, norm_iters)
        rg = orc.grad_support(X[k], Y[k], rows[s0:s1], cols[s0:s1], rv)
        ev = max(ev, normwise(vals[s0:s1], rv))
        el = max(el, abs(loss[k] - rl) / abs(rl))
        eg = max(eg, normwise(grad[k], rg))
    print(f"nnz {int(coo['nnz'])}: vals {ev:.2e} loss {el:.2e} grad {eg:.2e}")
    assert ev < TOL and el < TOL and eg < TOL, (ev, el, eg)


@pytest.mark.parametrize("norm_iters", [0, 5])
def test_apml_point_clouds(sot, orc, norm_iters):
    """The 8-cloud COO recipe at 2 clouds of 512 points, support at tau = 1e-8."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(5, B=2, n=512)
    check(sot, orc, X, Y, a, b, 5e-3, 300, 1e-8, 5e-3, norm_iters)


def test_apml_d8_weighted(sot, orc):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=300, m=270, d=8)
    check(sot, orc, X, Y, a, b, 0.1, 60, 1e-6, 0.1, 8, weighted=True)


def test_apml_every_pair_stored(sot, orc):
    """tau = 0 keeps every pair: the dense special case, ragged sizes."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=2, n=70, m=53)
    check(sot, orc, X, Y, a, b, 0.05, 40, 0.0, 0.05, 10)


def test_apml_many_columns(sot, orc):
    """More columns (m = 17000) than the row passes stage in shared memory
    (16384): the column maxima and sums go through global atomics instead;
    weighted, d = 3 (the support gradient fused into the last pass)."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=193, m=17000, d=3)
    check(sot, orc, X, Y, a, b, 0.1, 40, 1e-4, 0.1, 4, weighted=True)


def test_apml_gradient_unfused_d5(sot, orc):
    """d = 5: the support gradient runs as its own pass after the last one."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=2, n=150, m=161, d=5)
    check(sot, orc, X, Y, a, b, 0.2, 40, 1e-5, 0.2, 3, weighted=True)


def test_apml_rejects_invalid_support(sot):
    """An out-of-range column and unsorted rows are reported; every pass skips
    the bad indices, so nothing outside the arrays is touched first."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=1, n=64, m=60)
    Xd, Yd, _, _, coo = support(sot, X, Y, a, b, 0.05, 20, 1e-6, False)
    nnz = int(coo["nnz"])
    assert nnz > 4
    bad = dict(coo)
    bad["cols"] = coo["cols"].clone()
    bad["cols"][nnz // 2] = 60  # out of range
    with pytest.raises(sot.SotError) as ei:
        sot.sot_apml_coo(Xd, Yd, None, None, bad, 0.05, 3)
    assert ei.value.status == sot.SOT_ERR_INVALID_ARG
    bad = dict(coo)
    bad["rows"] = coo["rows"].flip(0).contiguous()  # rows descending
    with pytest.raises(sot.SotError) as ei:
        sot.sot_apml_coo(Xd, Yd, None, None, bad, 0.05, 3)
    assert ei.value.status == sot.SOT_ERR_INVALID_ARG
    # offsets that do not run from 0 to nnz, or decrease, are found on the device
    for off in ([0, nnz - 1], [0, nnz + 7]):
        bad = dict(coo)
        bad["batch_offsets"] = dev(np.array(off, dtype=np.int64))
        with pytest.raises(sot.SotError) as ei:
            sot.sot_apml_coo(Xd, Yd, None, None, bad, 0.05, 3)
        assert ei.value.status == sot.SOT_ERR_INVALID_ARG
    X3, Y3 = np.concatenate([X, X, X]), np.concatenate([Y, Y, Y])
    bad = {"rows": torch.cat([coo["rows"], coo["rows"]]), "cols": torch.cat([coo["cols"], coo["cols"]]),
           "batch_offsets": dev(np.array([0, nnz, nnz - 5, 2 * nnz], dtype=np.int64)), "nnz": 2 * nnz}
    with pytest.raises(sot.SotError) as ei:
        sot.sot_apml_coo(dev(X3), dev(Y3), None, None, bad, 0.05, 3)
    assert ei.value.status == sot.SOT_ERR_INVALID_ARG
    # the valid support still runs afterwards
    vals, loss, _ = sot.sot_apml_coo(Xd, Yd, None, None, coo, 0.05, 3, grad=False)
    torch.cuda.synchronize()
    assert np.all(np.isfinite(host(vals))) and np.isfinite(host(loss)).all()


def test_apml_full_workload_sampled_clouds(sot, orc):
    """The 8-cloud COO workload at full size (8 x 8192 points, the bench's
    support and 10 normalisations); the oracle follows clouds 0 and 7."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(5)
    Xd, Yd, _, _, coo = support(sot, X, Y, a, b, 5e-3, 300, 1e-8, False)
    vals, loss, grad = sot.sot_apml_coo(Xd, Yd, None, None, coo, 5e-3, 10)
    torch.cuda.synchronize()
    vals, loss, grad = host(vals), host(loss), host(grad)
    rows, cols = host(coo["rows"]).astype(np.int64), host(coo["cols"]).astype(np.int64)
    off = host(coo["batch_offsets"]).astype(np.int64)
    for k in (0, 7):
        s0, s1 = off[k], off[k + 1]
        rv, rl = orc.apml_coo(X[k], Y[k], None, None, rows[s0:s1], cols[s0:s1], 5e-3, 10)
        rg = orc.grad_support(X[k], Y[k], rows[s0:s1], cols[s0:s1], rv)
        ev, el, eg = normwise(vals[s0:s1], rv), abs(loss[k] - rl) / abs(rl), normwise(grad[k], rg)
        print(f"cloud {k}: nnz {s1 - s0} vals {ev:.2e} loss {el:.2e} grad {eg:.2e}")
        assert ev < TOL and el < TOL and eg < TOL, (k, ev, el, eg)


def test_apml_empty_row_and_column(sot, orc):
    """A support built by hand with every pair of row 5 and of column 7 left
    out (and the rest of two rows): empty rows and columns stay empty, the
    others are normalised as usual."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=1, n=40, m=36)
    rows, cols = np.divmod(np.arange(40 * 36), 36)
    keep = (rows != 5) & (cols != 7) & ~((rows == 9) & (cols > 3)) & ~((rows == 20) & (cols % 2 == 0))
    rows, cols = rows[keep].astype(np.int32), cols[keep].astype(np.int32)
    nnz = len(rows)
    coo = {"rows": dev(rows), "cols": dev(cols), "batch_offsets": dev(np.array([0, nnz], dtype=np.int64)),
           "nnz": nnz}
    vals, loss, grad = sot.sot_apml_coo(dev(X), dev(Y), None, None, coo, 0.05, 6)
    torch.cuda.synchronize()
    rv, rl = orc.apml_coo(X[0], Y[0], None, None, rows, cols, 0.05, 6)
    rg = orc.grad_support(X[0], Y[0], rows, cols, rv)
    ev, el, eg = normwise(host(vals), rv), abs(host(loss)[0] - rl) / abs(rl), normwise(host(grad)[0], rg)
    print(f"empty row/column: vals {ev:.2e} loss {el:.2e} grad {eg:.2e}")
    assert ev < TOL and el < TOL and eg < TOL, (ev, el, eg)
    assert np.all(host(grad)[0][5] == 0.0)
