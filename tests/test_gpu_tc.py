"""The tcgen05 tensor-core path (d = 64, fp16 x3 products) vs the fp64 oracle.

Reduced sizes span several 256-row blocks, several 128-column tiles and
ragged tails; the full n = m = 70000 configuration (the one bench.py times) is
checked on sampled rows of the first half-step, which the oracle computes
from X, Y and b alone, and on column marginals after 100 iterations.
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
    if s.sot_select_path(64, s.SOT_PREC_F16X3) != 2:
        pytest.skip("tensor-core path not built")
    return s


@pytest.mark.parametrize("n,m,B", [(1000, 1100, 1), (300, 257, 2), (513, 129, 1)])
def test_tc_matches_oracle(sot, orc, n, m, B):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=B, n=n, m=m, d=64)
    eps, iters = 0.1, 100
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    f, g = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=eps, iters_per_stage=iters, max_iters=iters,
                                 flags=sot.SOT_PREC_F16X3)
    c, gr, _ = sot.sot_plan_apply(Xd, Yd, ad, bd, f, g, eps)
    f, g, c, gr = host(f), host(g), host(c), host(gr)
    ef = eg = ec = egr = 0.0
    for k in range(B):
        fr, gref = orc.sinkhorn(X[k], Y[k], a[k], b[k], [eps], [iters])
        out = orc.plan_apply(X[k], Y[k], a[k], b[k], fr, gref, eps)
        e1, e2 = potentials_error(f[k:k + 1], g[k:k + 1], fr[None], gref[None])
        ef, eg = max(ef, e1), max(eg, e2)
        ec = max(ec, abs(c[k] - out["cost"]) / abs(out["cost"]))
        egr = max(egr, normwise(gr[k], out["grad"]))
    msg = f"f {ef:.2e} g {eg:.2e} cost {ec:.2e} grad {egr:.2e}"
    print(msg)
    assert max(ef, eg, ec, egr) < TOL, msg


def test_tc_agrees_with_fp32_path(sot):
    """Same problem through the fp16 x3 tensor path and the fp32 FMA path."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=3000, m=2600, d=64)
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    ft, gt = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=0.1, iters_per_stage=50, max_iters=50,
                                   flags=sot.SOT_PREC_F16X3)
    ff, gf = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=0.1, iters_per_stage=50, max_iters=50,
                                   flags=sot.SOT_PREC_FP32)
    ef, eg = potentials_error(host(ft), host(gt), host(ff), host(gf))
    assert ef < TOL and eg < TOL, (ef, eg)


def test_tc_full_size_first_half_step(sot, orc):
    """n = m = 70000, d = 64: after one iteration f is the first f-half, which
    the oracle evaluates row by row from X, Y and b (g = 0)."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4)
    eps = 0.1
    f, g = sot.sot_potentials(dev(X), dev(Y), dev(a), dev(b), eps=eps, iters=1)
    fh = host(f)[0]
    rows = np.random.default_rng(3).choice(X.shape[1], 48, replace=False)
    fr = orc.f_half(X[0][rows], Y[0], b[0], np.zeros(Y.shape[1]), eps)
    err = np.max(np.abs(fh[rows] - fr)) / np.max(np.abs(fr))
    assert err < TOL, err


def test_tc_full_size_screened_half_steps(sot, orc):
    """n = m = 70000, d = 64, as bench.py runs it: every warm half-step is a
    screened one.  Iteration 11 (both halves) is checked on sampled rows and
    columns against the oracle's half-steps from the potentials the GPU held
    after 10 iterations: the solve is bitwise reproducible, so the 11-iteration
    run passes through exactly those potentials."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4)
    eps = 0.1
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    sot.sot_profile_read_kinds()
    sot.sot_profile_enable(True)
    f10, g10 = sot.sot_potentials(Xd, Yd, ad, bd, eps=eps, iters=10)
    f11, g11 = sot.sot_potentials(Xd, Yd, ad, bd, eps=eps, iters=11)
    kinds = sot.sot_profile_read_kinds()
    sot.sot_profile_enable(False)
    assert kinds["screened"][0] == 18 + 20, kinds  # 9 + 10 warm iterations, two halves each
    g10h, f11h, g11h = host(g10)[0].astype(np.float64), host(f11)[0], host(g11)[0]
    rng = np.random.default_rng(11)
    rows = rng.choice(X.shape[1], 48, replace=False)
    cols = rng.choice(Y.shape[1], 48, replace=False)
    fr = orc.f_half(X[0][rows], Y[0], b[0], g10h, eps)
    gr = orc.g_half(X[0], Y[0][cols], a[0], f11h.astype(np.float64), eps)
    ef = np.max(np.abs(f11h[rows] - fr)) / np.max(np.abs(fr))
    eg = np.max(np.abs(g11h[cols] - gr)) / np.max(np.abs(gr))
    print(f"screened half-steps at full size: f {ef:.2e} g {eg:.2e}")
    assert ef < 1e-5 and eg < 1e-5, (ef, eg)


def test_tc_full_size_column_marginals(sot):
    """After 100 iterations (ending with a g-half) the column sums of the plan
    equal b exactly; recomputed in float64 for sampled columns."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4)
    eps = 0.1
    f, g = sot.sot_potentials(dev(X), dev(Y), dev(a), dev(b), eps=eps, iters=100)
    fh, gh = host(f)[0], host(g)[0]
    X64, Y64 = X[0].astype(np.float64), Y[0].astype(np.float64)
    a64, b64 = a[0].astype(np.float64), b[0].astype(np.float64)
    for j in np.random.default_rng(5).choice(Y.shape[1], 12, replace=False):
        C = ((X64 - Y64[j]) ** 2).sum(1)
        col = np.sum(a64 * b64[j] * np.exp((fh + gh[j] - C) / eps))
        assert abs(col - b64[j]) / b64[j] < 5e-3, (j, col / b64[j])


def test_tc_full_size_cost_gradient_and_error(sot, orc):
    """n = m = 70000, d = 64, as bench.py runs it: 100 iterations, then the
    cost and the gradient from the tensor-core plan application.  The oracle
    applies the plan of the GPU's own fp32 potentials over every pair
    ("FlashSinkhorn", Methodologie 3): cost and gradient (all rows) within
    1e-4, and the marginal error the solve reports equals the oracle's
    sum_i |sum_j P_ij - a_i| of the same potentials."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4)
    eps = 0.1
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    f, g, info = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=eps, iters_per_stage=100, max_iters=100, stats=True)
    c, gr, r = sot.sot_plan_apply(Xd, Yd, ad, bd, f, g, eps, rowsum=True)
    sot.sot_async_status()
    out = orc.plan_apply(X[0], Y[0], a[0], b[0], host(f)[0], host(g)[0], eps)
    ec = abs(host(c)[0] - out["cost"]) / abs(out["cost"])
    egr = normwise(host(gr)[0], out["grad"])
    er = normwise(host(r)[0], out["rowsum"])
    err_ref = float(np.sum(np.abs(out["rowsum"] - a[0].astype(np.float64))))
    print(f"70000 points: cost {ec:.2e} grad {egr:.2e} rowsum {er:.2e}; marginal error GPU {info['err'][0]:.4e} "
          f"oracle {err_ref:.4e}")
    assert ec < TOL and egr < TOL and er < TOL, (ec, egr, er)
    assert abs(info["err"][0] - err_ref) <= 1e-2 * err_ref + 1e-7, (info["err"][0], err_ref)


@pytest.mark.parametrize("n,m,B", [(1000, 1100, 1), (300, 257, 2)])
def test_tc_plan_apply_matches_oracle(sot, orc, n, m, B):
    """Cost, gradient and row sums from the tensor-core plan application, with
    the oracle's own potentials (rounded to fp32) as input."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=B, n=n, m=m, d=64)
    eps = 0.1
    fs, gs = [], []
    for k in range(B):
        fr, gref = orc.sinkhorn(X[k], Y[k], a[k], b[k], [eps], [60])
        fs.append(fr); gs.append(gref)
    f32 = np.stack(fs).astype(np.float32)
    g32 = np.stack(gs).astype(np.float32)
    c, gr, r = sot.sot_plan_apply(dev(X), dev(Y), dev(a), dev(b), dev(f32), dev(g32), eps, rowsum=True,
                                  flags=sot.SOT_PREC_F16X3)
    c, gr, r = host(c), host(gr), host(r)
    for k in range(B):
        out = orc.plan_apply(X[k], Y[k], a[k], b[k], f32[k], g32[k], eps)
        assert abs(c[k] - out["cost"]) / abs(out["cost"]) < TOL
        assert normwise(gr[k], out["grad"]) < TOL
        assert normwise(r[k], out["rowsum"]) < TOL


def test_tc_screened_agrees_with_full_half_steps(sot):
    """Warm half-steps screen pairs with hi*hi products and evaluate the kept
    ones exactly; the result equals the full half-steps' to well below the
    parity tolerance, and the screened kernel really ran."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=2, n=3000, m=2600, d=64)
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    sot.sot_profile_read_kinds()
    sot.sot_profile_enable(True)
    fs, gs = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=0.1, iters_per_stage=50, max_iters=50,
                                   flags=sot.SOT_PREC_F16X3)
    kinds = sot.sot_profile_read_kinds()
    ff, gf = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=0.1, iters_per_stage=50, max_iters=50,
                                   flags=sot.SOT_PREC_F16X3 | sot.SOT_TC_NO_SCREEN)
    kinds_full = sot.sot_profile_read_kinds()
    sot.sot_profile_enable(False)
    assert kinds["screened"][0] == 98 and kinds["full"][0] == 2, kinds  # the cold first iteration is full
    assert kinds_full["screened"][0] == 0 and kinds_full["full"][0] == 100, kinds_full
    ef, eg = potentials_error(host(fs), host(gs), host(ff), host(gf))
    assert ef < 2e-5 and eg < 2e-5, (ef, eg)


def test_tc_screen_gives_way_on_a_dense_plan(sot, orc):
    """At a large eps every column of a row is within reach of its sum: the
    candidate lists overflow, those rows take the exact full-row LSE, and the
    solver continues with full half-steps.  Results still match the oracle."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=600, m=500, d=64)
    eps, iters = 200.0, 12
    sot.sot_profile_read_kinds()
    sot.sot_profile_enable(True)
    f, g = sot.sot_potentials_ex(dev(X), dev(Y), dev(a), dev(b), eps=eps, iters_per_stage=iters, max_iters=iters,
                                 flags=sot.SOT_PREC_F16X3)
    kinds = sot.sot_profile_read_kinds()
    sot.sot_profile_enable(False)
    assert kinds["screened"][0] == 2, kinds  # one screened iteration, then full half-steps
    fr, gref = orc.sinkhorn(X[0], Y[0], a[0], b[0], [eps], [iters])
    ef, eg = potentials_error(host(f), host(g), fr[None], gref[None])
    assert ef < TOL and eg < TOL, (ef, eg)


def test_tc_screened_annealed_schedule(sot, orc):
    """Screening across eps stages (each stage's first iteration is full, the
    bounds restart): eps 1 -> 0.1 by x0.5, 10 iterations per stage."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=1500, m=1300, d=64)
    f, g, info = sot.sot_potentials_ex(dev(X), dev(Y), dev(a), dev(b), eps=0.1, eps_init=1.0, eps_factor=0.5,
                                       iters_per_stage=10, max_iters=0, flags=sot.SOT_PREC_F16X3, stats=True)
    stages = orc.anneal_stages(1.0, 0.5, 0.1)
    assert info["stages_done"] == len(stages)
    fr, gref = orc.sinkhorn(X[0], Y[0], a[0], b[0], stages, [10] * len(stages))
    ef, eg = potentials_error(host(f), host(g), fr[None], gref[None])
    assert ef < TOL and eg < TOL, (ef, eg)


@pytest.mark.parametrize("d,n,m,eps", [(128, 1100, 1000, 0.2), (192, 600, 520, 0.3), (256, 700, 650, 0.4),
                                       (512, 600, 520, 0.8), (1024, 400, 300, 1.6)])
def test_tc_wide_matches_oracle(sot, orc, d, n, m, eps):
    """d = 128, 192, 256, 512 and 1024 on the tensor path ("FlashSinkhorn",
    Experimentele Resultaten: the streaming kernels run up to d = 1024): warm
    half-steps on the screened kernel with a K loop over slices of 64 (at 512
    and 1024 the row tiles' slices stream with the column tiles'), cold
    half-steps and the plan application on the fp32 kernels.  Gaussian recipe with softmax
    weights; potentials, cost and gradient against the oracle."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=n, m=m, d=d)
    iters = 60
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    assert sot.sot_select_path(d, 0) == 2
    sot.sot_profile_read_kinds()
    sot.sot_profile_enable(True)
    f, g = sot.sot_potentials(Xd, Yd, ad, bd, eps=eps, iters=iters)
    kinds = sot.sot_profile_read_kinds()
    sot.sot_profile_enable(False)
    assert kinds["screened"][0] == 2 * iters - 2, kinds  # the cold first iteration is dense
    c, gr, _ = sot.sot_plan_apply(Xd, Yd, ad, bd, f, g, eps)
    fr, gref = orc.sinkhorn(X[0], Y[0], a[0], b[0], [eps], [iters])
    ef, eg = potentials_error(host(f), host(g), fr[None], gref[None])
    out = orc.plan_apply(X[0], Y[0], a[0], b[0], host(f)[0], host(g)[0], eps)
    ec = abs(host(c)[0] - out["cost"]) / abs(out["cost"])
    egr = normwise(host(gr)[0], out["grad"])
    msg = f"d = {d}: f {ef:.2e} g {eg:.2e} cost {ec:.2e} grad {egr:.2e}"
    print(msg)
    assert max(ef, eg, ec, egr) < TOL, msg


def test_tc_wide_screened_agrees_with_fp32(sot):
    """d = 128, 256 and 512 with two clouds: the tensor path and the fp32 path
    give the same potentials to well below the parity tolerance."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    for d, eps in ((128, 0.2), (256, 0.4), (512, 0.8)):
        X, Y, a, b = dg.make_batch(4, B=2, n=1500, m=1300, d=d)
        Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
        ft, gt = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=eps, iters_per_stage=40, max_iters=40,
                                       flags=sot.SOT_PREC_F16X3)
        ff, gf = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=eps, iters_per_stage=40, max_iters=40,
                                       flags=sot.SOT_PREC_FP32)
        ef, eg = potentials_error(host(ft), host(gt), host(ff), host(gf))
        assert ef < 2e-5 and eg < 2e-5, (d, ef, eg)


@pytest.mark.parametrize("d,n,m,eps,forced", [(17, 700, 650, 0.03, False), (100, 600, 520, 0.16, False),
                                              (300, 500, 450, 0.47, False), (700, 400, 300, 1.1, False),
                                              (8, 700, 650, 0.0125, True)])
def test_tc_padded_dims_match_oracle(sot, orc, d, n, m, eps, forced):
    """Dimensions the tensor cores do not take natively run there with the
    coordinates zero-padded (17 -> 64, 100 -> 128, 300 -> 512, 700 -> 1024;
    d = 8 with the fp16 split forced): potentials, cost and gradient (at the
    caller's d) against the oracle."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=n, m=m, d=d)
    flags = sot.SOT_PREC_F16X3 if forced else 0
    assert sot.sot_select_path(d, flags) == 2
    Xd, Yd, ad, bd = dev(X), dev(Y), dev(a), dev(b)
    iters = 60
    f, g = sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=eps, iters_per_stage=iters, max_iters=iters, flags=flags)
    c, gr, _ = sot.sot_plan_apply(Xd, Yd, ad, bd, f, g, eps, flags=flags)
    assert tuple(gr.shape) == (1, n, d)
    fr, gref = orc.sinkhorn(X[0], Y[0], a[0], b[0], [eps], [iters])
    ef, eg = potentials_error(host(f), host(g), fr[None], gref[None])
    out = orc.plan_apply(X[0], Y[0], a[0], b[0], host(f)[0], host(g)[0], eps)
    ec = abs(host(c)[0] - out["cost"]) / abs(out["cost"])
    egr = normwise(host(gr)[0], out["grad"])
    msg = f"d = {d}: f {ef:.2e} g {eg:.2e} cost {ec:.2e} grad {egr:.2e}"
    print(msg)
    assert max(ef, eg, ec, egr) < TOL, msg
