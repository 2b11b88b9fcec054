"""Thresholded COO plan and the gradient on its support, GPU vs oracle
("From Theory to Throughput: CUDA-Optimized APML", Abstract / Innovation).

Gate A (bit-exact): the library reports the fp32 operands its predicate reads
(sot_plan_coo_operands); a CPU fp32 replica of the predicate
(tests/coo_replica.c, not the oracle) recomputes the row and column maxima
from them, which must equal the GPU's bit for bit, and the support, whose
row and column index lists must equal the GPU's exactly.

Gate B (end-to-end): the fp64 oracle decides from its own fp64 potentials;
the GPU decides from those potentials rounded to fp32.  Every pair whose
log-margin to the threshold exceeds a band delta must be decided the same way,
with delta derived from the data: three times the exponent error that
rounding the potentials causes, (max|df| + max|dg|) / eps, plus a bound on the
fp32 score's own rounding, 16 u (|bias| + kappa (|x| + |y|)^2 + |max| +
|log2 tau|) ln 2 with u = 2^-24 (each of the ~10 rounded steps of a score
and of its threshold contributes at most u times a term of that size).  The
pairs inside the band are counted and must stay below 0.1 % of the stored
entries.  Values within 1e-4 relative; support gradients within 1e-4.
"""
import numpy as np
import pytest

import coo_replica
from gpu_util import TOL, dev, host, normwise

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

U32 = 2.0 ** -24
INBAND_MAX = 1e-3  # in-band pairs per stored entry


@pytest.fixture(scope="module")
def sot():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sinkhorn_point_cloud_gb300 as s
    from sinkhorn_point_cloud_gb300 import build
    build.build()
    return s


def _problem(orc, n=1024, B=2, eps=5e-3, iters=300):
    """The 8-cloud sphere recipe reduced to B clouds of n points; the oracle's
    fp64 potentials after `iters` iterations."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(5, B=B, n=n)
    fs, gs = [], []
    for k in range(B):
        f, g = orc.sinkhorn(X[k], Y[k], None, None, [eps], [iters])
        fs.append(f); gs.append(g)
    f64, g64 = np.stack(fs), np.stack(gs)
    return X, Y, f64.astype(np.float32), g64.astype(np.float32), eps, f64, g64


@pytest.fixture(scope="module")
def prob(orc):
    return _problem(orc)


def _f32(t):
    return t.detach().cpu().numpy().astype(np.float32)


def _same_bits(a, b):
    a = np.ascontiguousarray(a, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    return a.shape == b.shape and np.array_equal(a.view(np.uint32), b.view(np.uint32))


def gate_a(sot, X, Y, a, b, f, g, eps, tau, dirs, clouds=None):
    """Gate A on the given device inputs; returns the GPU's COO."""
    ops = sot.sot_plan_coo_operands(X, Y, a, b, f, g, eps, threshold=tau)
    out = sot.sot_plan_coo(X, Y, a, b, f, g, eps, threshold=tau, dirs=dirs)
    off = host(out["batch_offsets"]).astype(np.int64)
    rows, cols = out["rows"].cpu().numpy(), out["cols"].cpu().numpy()
    B = X.shape[0]
    for k in (range(B) if clouds is None else clouds):
        rep = coo_replica.replica(_f32(ops["xc"][k]), _f32(ops["lwx"][k]), _f32(ops["Lx"][k]), _f32(ops["yc"][k]),
                                  _f32(ops["lwy"][k]), _f32(ops["Ly"][k]), ops["kappa"], ops["log2tau"], dirs)
        assert _same_bits(_f32(ops["Mr"][k]), rep["Mr"]), f"cloud {k}: row maxima differ from the fp32 replica"
        assert _same_bits(_f32(ops["Mc"][k]), rep["Mc"]), f"cloud {k}: column maxima differ from the fp32 replica"
        r, c = rows[off[k]:off[k + 1]], cols[off[k]:off[k + 1]]
        assert len(r) == len(rep["rows"]), f"cloud {k}: {len(r)} entries, replica {len(rep['rows'])}"
        assert np.array_equal(r, rep["rows"]) and np.array_equal(c, rep["cols"]), f"cloud {k}: index lists differ"
    return out, ops


def rounding_band(ops, k, d):
    """Bound on the fp32 score's own rounding, in natural-log units (see the
    module docstring)."""
    xc, yc = _f32(ops["xc"][k]).astype(np.float64), _f32(ops["yc"][k]).astype(np.float64)
    bias = np.max(np.abs(_f32(ops["lwy"][k]) - _f32(ops["Ly"][k]))) + \
        np.max(np.abs(_f32(ops["lwx"][k]) - _f32(ops["Lx"][k])))
    rad = np.sqrt((xc ** 2).sum(1)).max() + np.sqrt((yc ** 2).sum(1)).max()
    mx = max(np.max(np.abs(_f32(ops["Mr"][k]))), np.max(np.abs(_f32(ops["Mc"][k]))))
    lt = abs(ops["log2tau"]) if np.isfinite(ops["log2tau"]) else 0.0
    return 16 * U32 * (bias + ops["kappa"] * rad * rad + mx + lt) * np.log(2.0)


@pytest.mark.parametrize("dirs", [1, 2, 3])
def test_coo_gate_a_bit_exact(sot, prob, dirs):
    """The GPU's own potentials (300 iterations of the reduced recipe)."""
    X, Y, _, _, eps, _, _ = prob
    Xd, Yd = dev(X), dev(Y)
    f, g = sot.sot_potentials(Xd, Yd, eps=eps, iters=300)
    gate_a(sot, Xd, Yd, None, None, f, g, eps, 1e-8, dirs)


@pytest.mark.parametrize("d,tau", [(2, 1e-8), (8, 1e-8), (8, 1e-3), (64, 1e-8), (512, 1e-8)])
def test_coo_gate_a_other_layouts(sot, d, tau):
    """Weighted clouds in d = 2 (point layout) and d = 8, 64, 512 (the dense
    layout's expanded-form scores; at 512 the maxima pass streams the
    coordinates in slices); potentials from a GPU solve."""
    rng = np.random.default_rng(100 + d)
    B, n, m = 2, 700, 650
    X = rng.normal(size=(B, n, d)).astype(np.float32)
    Y = (rng.normal(size=(B, m, d)) + 0.3).astype(np.float32)
    a = rng.random((B, n)) + 0.1
    b = rng.random((B, m)) + 0.1
    a = (a / a.sum(1, keepdims=True)).astype(np.float32)
    b = (b / b.sum(1, keepdims=True)).astype(np.float32)
    eps = 0.05 * d
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    f, g = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=eps, iters_per_stage=50, flags=sot.SOT_PREC_FP32)[:2]
    gate_a(sot, Xd, Yd, ad, bd, f, g, eps, tau, 3)


@pytest.mark.parametrize("dirs", [1, 2, 3])
def test_coo_gate_b_band(sot, orc, prob, dirs):
    X, Y, f, g, eps, f64, g64 = prob
    Xd, Yd, fd, gd = dev(X), dev(Y), dev(f), dev(g)
    ops = sot.sot_plan_coo_operands(Xd, Yd, None, None, fd, gd, eps, threshold=1e-8)
    out = sot.sot_plan_coo(Xd, Yd, None, None, fd, gd, eps, threshold=1e-8, dirs=dirs)
    rows, cols, vals, off = host(out["rows"]).astype(int), host(out["cols"]).astype(int), host(out["vals"]), \
        host(out["batch_offsets"]).astype(int)
    assert off[0] == 0 and off[-1] == out["nnz"]
    total_inband = 0
    for k in range(X.shape[0]):
        s0, s1 = off[k], off[k + 1]
        r, c = rows[s0:s1], cols[s0:s1]
        key = r.astype(np.int64) * Y.shape[1] + c
        assert np.all(np.diff(key) > 0), "not row-major ascending within the cloud"
        pot = (np.max(np.abs(f[k] - f64[k])) + np.max(np.abs(g[k] - g64[k]))) / eps
        band = 3 * pot + rounding_band(ops, k, X.shape[2])
        assert band < 1e-2, band
        ref = orc.coo(X[k], Y[k], None, None, f64[k], g64[k], eps, 1e-8, dirs, band=band)
        sure = ref["margins"] > band
        want = set(zip(ref["rows"][sure].tolist(), ref["cols"][sure].tolist()))
        allowed = set(zip(ref["rows"].tolist(), ref["cols"].tolist()))  # margin >= -band
        got = set(zip(r.tolist(), c.tolist()))
        assert not (want - got), f"{len(want - got)} pairs above the band missing"
        assert not (got - allowed), f"{len(got - allowed)} pairs below the band stored"
        inband = int(np.sum(np.abs(ref["margins"]) <= band))
        assert inband <= INBAND_MAX * (s1 - s0), f"{inband} in-band pairs of {s1 - s0} (band {band:.2e})"
        total_inband += inband
        # values on the pairs both sides store
        keep = ref["margins"] >= 0
        refmap = dict(zip(zip(ref["rows"][keep].tolist(), ref["cols"][keep].tolist()), ref["vals"][keep].tolist()))
        common = [(i, j, v) for i, j, v in zip(r.tolist(), c.tolist(), vals[s0:s1].tolist()) if (i, j) in refmap]
        gv = np.array([v for _, _, v in common])
        rv = np.array([refmap[(i, j)] for i, j, _ in common])
        assert normwise(gv, rv) < TOL
    print("in-band pairs:", total_inband, "nnz:", out["nnz"])


def test_coo_threshold_limits(sot, orc, prob):
    X, Y, f, g, eps = prob[:5]
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
    X, Y, f, g, eps = prob[:5]
    with pytest.raises(sot.SotError) as ei:
        sot.sot_plan_coo(dev(X), dev(Y), None, None, dev(f), dev(g), eps, threshold=1e-8, dirs=3, capacity=5)
    assert ei.value.status == sot.SOT_ERR_CAPACITY


def test_grad_on_given_support(sot, orc, prob):
    """The support gradient of the oracle's COO, computed on the GPU."""
    X, Y, f, g, eps = prob[:5]
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
    """The GPU's support and values from fp32 potentials against the oracle's
    support gradient from the same potentials: the supports differ only in
    pairs near the threshold (P_ij ~ 1e-8 of a row's largest entry), and the
    values carry float-float exponents."""
    X, Y, f, g, eps = prob[:5]
    out = sot.sot_plan_coo(dev(X), dev(Y), None, None, dev(f), dev(g), eps, threshold=1e-8, dirs=3)
    gr = host(sot.sot_grad_x_coo(dev(X), dev(Y), out["rows"], out["cols"], out["vals"], out["batch_offsets"]))
    for k in range(X.shape[0]):
        ref = orc.coo(X[k], Y[k], None, None, f[k], g[k], eps, 1e-8, 3)
        gref = orc.grad_support(X[k], Y[k], ref["rows"], ref["cols"], ref["vals"])
        assert normwise(gr[k], gref) < TOL


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
    configuration).  Gate A on clouds 0 and 7; beyond it, checked here:
    row-major order, every row keeps its argmax, column sums of the dense plan
    (exact after a g-half) and the kept mass of sampled rows, all recomputed
    in float64 from the GPU's potentials."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(5)
    Xd, Yd = dev(X), dev(Y)
    eps = 5e-3
    f, g = sot.sot_potentials(Xd, Yd, eps=eps, iters=300)
    # Gate A at full size on clouds 0 and 7 (the replica takes ~1 s per cloud)
    out, _ = gate_a(sot, Xd, Yd, None, None, f, g, eps, 1e-8, 3, clouds=(0, 7))
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
