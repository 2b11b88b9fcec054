"""Thresholded COO plan and the gradient on its support, GPU vs oracle.

Given the same float32 potentials, every pair whose log-margin to the
threshold exceeds the rounding band of the fp32 score must be decided the
same way (indices exact); pairs inside the band may go either way and are
counted.  Values within 1e-4 relative; support gradients within 1e-4.
"""
import numpy as np
import pytest

from gpu_util import TOL, dev, host, normwise

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

BAND = 2e-3  # natural-log units; fp32 score rounding at these magnitudes is ~2e-4


@pytest.fixture(scope="module")
def sot():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sinkhorn_point_cloud_gb300 as s
    from sinkhorn_point_cloud_gb300 import build
    build.build()
    return s


def _problem(orc, n=1024, B=2, eps=5e-3, iters=300):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(5, B=B, n=n)
    fs, gs = [], []
    for k in range(B):
        f, g = orc.sinkhorn(X[k], Y[k], None, None, [eps], [iters])
        fs.append(f); gs.append(g)
    return X, Y, np.stack(fs).astype(np.float32), np.stack(gs).astype(np.float32), eps


@pytest.fixture(scope="module")
def prob(orc):
    return _problem(orc)


def _compare(got_rows, got_cols, ref):
    """Band comparison of one cloud: returns (#in-band pairs, #disagreements outside the band)."""
    sure = ref["margins"] > BAND
    want = set(zip(ref["rows"][sure].tolist(), ref["cols"][sure].tolist()))
    allowed = set(zip(ref["rows"].tolist(), ref["cols"].tolist()))  # margin >= -BAND
    got = set(zip(got_rows.tolist(), got_cols.tolist()))
    bad = len(want - got) + len(got - allowed)
    inband = int(np.sum(np.abs(ref["margins"]) <= BAND))
    return inband, bad


@pytest.mark.parametrize("dirs", [1, 2, 3])
def test_coo_indices_match_outside_rounding_band(sot, orc, prob, dirs):
    X, Y, f, g, eps = prob
    out = sot.sot_plan_coo(dev(X), dev(Y), None, None, dev(f), dev(g), eps, threshold=1e-8, dirs=dirs)
    rows, cols, vals, off = host(out["rows"]).astype(int), host(out["cols"]).astype(int), host(out["vals"]), \
        host(out["batch_offsets"]).astype(int)
    assert off[0] == 0 and off[-1] == out["nnz"]
    total_inband = 0
    for k in range(X.shape[0]):
        s0, s1 = off[k], off[k + 1]
        r, c = rows[s0:s1], cols[s0:s1]
        key = r.astype(np.int64) * Y.shape[1] + c
        assert np.all(np.diff(key) > 0), "not row-major ascending within the cloud"
        ref = orc.coo(X[k], Y[k], None, None, f[k], g[k], eps, 1e-8, dirs, band=BAND)
        inband, bad = _compare(r, c, ref)
        assert bad == 0, f"{bad} pairs decided differently outside the band"
        total_inband += inband
        # values on the common pairs
        sure = ref["margins"] >= 0
        refmap = dict(zip(zip(ref["rows"][sure].tolist(), ref["cols"][sure].tolist()), ref["vals"][sure].tolist()))
        common = [(i, j, v) for i, j, v in zip(r.tolist(), c.tolist(), vals[s0:s1].tolist()) if (i, j) in refmap]
        gv = np.array([v for _, _, v in common])
        rv = np.array([refmap[(i, j)] for i, j, _ in common])
        assert normwise(gv, rv) < TOL
    print("in-band pairs:", total_inband, "nnz:", out["nnz"])


def test_coo_threshold_limits(sot, orc, prob):
    X, Y, f, g, eps = prob
    n, m = X.shape[1], Y.shape[1]
    full = sot.sot_plan_coo(dev(X), dev(Y), None, None, dev(f), dev(g), eps, threshold=0.0, dirs=3)
    assert full["nnz"] == X.shape[0] * n * m
    assert np.array_equal(host(full["batch_offsets"]).astype(int), np.arange(X.shape[0] + 1) * n * m)
    top = sot.sot_plan_coo(dev(X), dev(Y), None, None, dev(f), dev(g), eps, threshold=1.0, dirs=1)
    r = host(top["rows"]).astype(int)
    off = host(top["batch_offsets"]).astype(int)
    for k in range(X.shape[0]):
        assert np.array_equal(np.unique(r[off[k]:off[k + 1]]), np.arange(n)), "tau = 1 keeps each row's argmax"


def test_coo_capacity_error(sot, prob):
    X, Y, f, g, eps = prob
    with pytest.raises(sot.SotError) as ei:
        sot.sot_plan_coo(dev(X), dev(Y), None, None, dev(f), dev(g), eps, threshold=1e-8, dirs=3, capacity=5)
    assert ei.value.status == sot.SOT_ERR_CAPACITY


def test_grad_on_given_support(sot, orc, prob):
    """The support gradient of the oracle's COO, computed on the GPU."""
    X, Y, f, g, eps = prob
    rows, cols, vals, offs = [], [], [], [0]
    refs = []
    for k in range(X.shape[0]):
        ref = orc.coo(X[k], Y[k], None, None, f[k], g[k], eps, 1e-8, 3)
        rows.append(ref["rows"]); cols.append(ref["cols"]); vals.append(ref["vals"].astype(np.float32))
        offs.append(offs[-1] + len(ref["rows"]))
        refs.append(orc.grad_support(X[k], Y[k], ref["rows"], ref["cols"], ref["vals"].astype(np.float32)))
    R = dev(np.concatenate(rows).astype(np.int32))
    Cc = dev(np.concatenate(cols).astype(np.int32))
    V = dev(np.concatenate(vals))
    O = dev(np.array(offs, dtype=np.int64))
    gr = host(sot.sot_grad_x_coo(dev(X), dev(Y), R, Cc, V, O))
    for k in range(X.shape[0]):
        assert normwise(gr[k], refs[k]) < TOL


def test_grad_on_own_support_end_to_end(sot, orc, prob):
    X, Y, f, g, eps = prob
    out = sot.sot_plan_coo(dev(X), dev(Y), None, None, dev(f), dev(g), eps, threshold=1e-8, dirs=3)
    gr = host(sot.sot_grad_x_coo(dev(X), dev(Y), out["rows"], out["cols"], out["vals"], out["batch_offsets"]))
    for k in range(X.shape[0]):
        ref = orc.coo(X[k], Y[k], None, None, f[k], g[k], eps, 1e-8, 3)
        gref = orc.grad_support(X[k], Y[k], ref["rows"], ref["cols"], ref["vals"])
        assert normwise(gr[k], gref) < 1e-3


def test_grad_coo_rejects_bad_input(sot):
    X = np.zeros((1, 4, 3), np.float32)
    Y = np.ones((1, 5, 3), np.float32)
    rows = dev(np.array([1, 0, 2], np.int32))  # not sorted
    cols = dev(np.array([0, 1, 2], np.int32))
    vals = dev(np.ones(3, np.float32))
    off = dev(np.array([0, 3], np.int64))
    with pytest.raises(sot.SotError) as ei:
        sot.sot_grad_x_coo(dev(X), dev(Y), rows, cols, vals, off)
    assert ei.value.status == sot.SOT_ERR_INVALID_ARG
    rows = dev(np.array([0, 1, 2], np.int32))
    cols = dev(np.array([0, 7, 2], np.int32))  # column out of range (skipped, flagged)
    with pytest.raises(sot.SotError):
        sot.sot_grad_x_coo(dev(X), dev(Y), rows, cols, vals, off)


def test_check_inputs(sot):
    X = np.random.default_rng(0).random((1, 10, 3)).astype(np.float32)
    assert sot.sot_check_inputs(dev(X), dev(X)) == sot.SOT_OK
    Xb = X.copy()
    Xb[0, 3, 1] = np.nan
    assert sot.sot_check_inputs(dev(Xb), dev(X)) == sot.SOT_ERR_NONFINITE
    a = np.full((1, 10), 0.1, np.float32)
    a[0, 2] = 0.0
    assert sot.sot_check_inputs(dev(X), dev(X), dev(a), None) == sot.SOT_ERR_NONFINITE


def test_workload5_full_size_properties(sot):
    """B=8, n=m=8192, eps=5e-3, 300 iterations, then the COO (the timed
    configuration).  At this size the oracle cannot follow; checked here:
    row-major order, every row keeps its argmax, column sums of the dense plan
    (exact after a g-half) and the kept mass of sampled rows, all recomputed
    in float64 from the GPU's potentials."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(5)
    Xd, Yd = dev(X), dev(Y)
    eps = 5e-3
    f, g = sot.sot_potentials(Xd, Yd, eps=eps, iters=300)
    out = sot.sot_plan_coo(Xd, Yd, None, None, f, g, eps, threshold=1e-8, dirs=3)
    off = host(out["batch_offsets"]).astype(np.int64)
    rows = host(out["rows"]).astype(np.int64)
    cols = host(out["cols"]).astype(np.int64)
    fh, gh = host(f), host(g)
    rng = np.random.default_rng(7)
    n = X.shape[1]
    for k in (0, 7):
        r, c = rows[off[k]:off[k + 1]], cols[off[k]:off[k + 1]]
        key = r * n + c
        assert np.all(np.diff(key) > 0)
        assert np.array_equal(np.unique(r), np.arange(n))
        X64, Y64 = X[k].astype(np.float64), Y[k].astype(np.float64)
        for j in rng.choice(n, 8, replace=False):
            C = ((X64 - Y64[j]) ** 2).sum(1)
            colsum = np.sum(np.exp((fh[k] + gh[k, j] - C) / eps) / (n * n))
            assert abs(colsum - 1.0 / n) < 2e-3 / n, colsum * n
