"""eps-annealing and the marginal-error stop test on the GPU vs the oracle.

The stop rule is the reading in include/sot.h (sot_schedule): the test runs
after every iteration at the final eps (or in every stage with early exit).
fp32 and fp64 may pass the threshold on different iterations, so the parity
of the potentials is taken in replay mode: the oracle runs the GPU's realised
schedule (its stage eps values, rounded to fp32 as the GPU holds them, and
its per-stage iteration counts) and the potentials must agree within the
usual 1e-4.  Separately, the realised counts are compared with the oracle's
own stop with a small allowance, and the oracle's marginal error after the
replay must be below the tolerance.
"""
import json
import os

import numpy as np
import pytest

from gpu_util import TOL, dev, host, potentials_error

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


def replay_schedule(orc, info, eps0=1.0, factor=0.9, eps_min=1e-3):
    """The GPU's realised schedule: (eps of each stage entered, as fp32, and its iterations)."""
    stages = orc.anneal_stages(eps0, factor, eps_min)[: info["stages_done"]]
    return stages.astype(np.float32).astype(np.float64), np.array(info["stage_iters"], dtype=np.int64)


def test_workload3_reduced_annealed_stop(sot, orc):
    """GMM clouds, eps 1 -> 1e-3 by x0.9 per stage, 20 iterations per stage,
    stop at marginal error < 1e-4 (n = m = 512, 2 clouds)."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(3, B=2, n=512)
    f, g, info = sot.sot_potentials_ex(dev(X), dev(Y), eps=1e-3, eps_init=1.0, eps_factor=0.9, iters_per_stage=20,
                                       max_iters=5000, tol=1e-4, stats=True)
    assert info["stages_done"] == 67, info["stages_done"]
    assert info["stage_iters"][:66] == [20] * 66
    assert info["converged"], info
    assert max(info["err"]) < 1e-4
    # iteration count against the oracle's own stop (the batch stops on its worst cloud)
    its = []
    for k in range(2):
        out = orc.sinkhorn_anneal(X[k], Y[k], None, None, 1.0, 0.9, 1e-3, 20, 1e-4, 5000)
        its.append(out["iters_done"])
        assert out["converged"]
    ref_iters = max(its)
    assert abs(info["iters_done"] - ref_iters) <= max(3, 0.02 * ref_iters), (info["iters_done"], its)
    # potentials in replay mode, every cloud
    eps_list, iters_list = replay_schedule(orc, info)
    fh, gh = host(f), host(g)
    for k in range(2):
        fr, gr = orc.sinkhorn(X[k], Y[k], None, None, eps_list, iters_list)
        ef, eg = potentials_error(fh[k:k + 1], gh[k:k + 1], fr[None], gr[None])
        assert ef < TOL and eg < TOL, (k, ef, eg)
        e_replay = orc.marginal_err(X[k], Y[k], None, None, fr, gr, eps_list[-1])
        assert e_replay < 1e-4 or abs(e_replay - info["err"][k]) <= 0.1 * e_replay, (k, e_replay, info["err"][k])


def test_workload3_full_size_final_iteration(sot, orc):
    """The 4-cloud GMM workload at full size (n = m = 16384) with its annealed
    schedule, as bench.py runs it.  Checked against the oracle on cloud 0:
    the final iteration's f-half (sampled rows, from the g the GPU held one
    iteration earlier: the solve is bitwise reproducible, so the run capped
    one iteration sooner ends there) and g-half (sampled columns, from the
    final f); and the marginal error the solve reports, against the oracle's
    definition evaluated on the GPU's final potentials (every pair), which
    also records whether the run met the stop test."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(3)
    Xd, Yd = dev(X), dev(Y)
    kw = dict(eps=1e-3, eps_init=1.0, eps_factor=0.9, iters_per_stage=20, tol=1e-4, stats=True)
    f, g, info = sot.sot_potentials_ex(Xd, Yd, max_iters=5000, **kw)
    N = info["iters_done"]
    f0, g0, info0 = sot.sot_potentials_ex(Xd, Yd, max_iters=N - 1, **kw)
    assert info0["iters_done"] == N - 1
    eps = info["final_eps"]
    fN, gN, gprev = host(f)[0], host(g)[0], host(g0)[0]
    rng = np.random.default_rng(31)
    rows = rng.choice(X.shape[1], 64, replace=False)
    cols = rng.choice(Y.shape[1], 64, replace=False)
    fr = orc.f_half(X[0][rows], Y[0], None, gprev, eps)
    gr = orc.g_half(X[0], Y[0][cols], None, fN, eps)
    scale = max(np.max(np.abs(fr)), np.max(np.abs(gr)))
    ef = np.max(np.abs(fN[rows] - fr)) / scale
    eg = np.max(np.abs(gN[cols] - gr)) / scale
    err_ref = orc.marginal_err(X[0], Y[0], None, None, fN, gN, eps)
    print(f"16384 points, {N} iterations, converged {info['converged']}: last f-half {ef:.2e}, g-half {eg:.2e}; "
          f"marginal error GPU {info['err'][0]:.4e} oracle {err_ref:.4e}")
    assert ef < TOL and eg < TOL, (ef, eg)
    assert abs(info["err"][0] - err_ref) <= 0.1 * err_ref + 1e-7, (info["err"][0], err_ref)
    assert info["converged"] == (max(info["err"]) < 1e-4)


def test_early_exit_matches_oracle_schedule(sot, orc):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(3, B=1, n=300, m=280)
    f, g, info = sot.sot_potentials_ex(dev(X), dev(Y), eps=0.02, eps_init=0.5, eps_factor=0.5, iters_per_stage=40,
                                       max_iters=2000, tol=1e-3, flags=sot.SOT_STAGE_EARLY_EXIT, stats=True)
    out = orc.sinkhorn_anneal(X[0], Y[0], None, None, 0.5, 0.5, 0.02, 40, 1e-3, 2000, early_exit=True)
    assert info["stages_done"] == out["stages_done"]
    gi, oi = np.array(info["stage_iters"]), out["stage_iters"]
    assert np.all(np.abs(gi - oi) <= 2), (gi, oi)


def test_fixed_schedule_stats(sot, orc):
    """A fixed schedule reports its iterations and the marginal error of the
    returned iterate, which agrees with the oracle's definition."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=400, m=350, d=8)
    f, g, info = sot.sot_potentials_ex(dev(X), dev(Y), dev(a), dev(b), eps=0.5, iters_per_stage=30, max_iters=30,
                                       stats=True)
    assert info["iters_done"] == 30 and info["stages_done"] == 1 and not info["converged"]
    fr, gr = orc.sinkhorn(X[0], Y[0], a[0], b[0], [0.5], [30])
    e_ref = orc.marginal_err(X[0], Y[0], a[0], b[0], fr, gr, 0.5)
    assert abs(info["err"][0] - e_ref) <= 1e-3 * e_ref + 1e-6, (info["err"][0], e_ref)


def test_max_iters_cap_without_convergence(sot):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(3, B=1, n=256)
    f, g, info = sot.sot_potentials_ex(dev(X), dev(Y), eps=1e-3, iters_per_stage=5, max_iters=12, tol=1e-12,
                                       stats=True)
    assert info["iters_done"] == 12 and not info["converged"]
    assert np.isfinite(info["err"][0])


RECORD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "anneal_gmm8_n16384_cloud0.json")


def test_workload3_full_size_against_oracle_record(sot):
    """Cloud 0 of the 4-cloud Gaussian-mixture workload at full size (n = m =
    16384) on its annealed schedule (eps 1 -> 1e-3 by x0.9 per stage, 20
    iterations per stage, stop at a marginal error below 1e-4, at most 5000
    iterations) against the oracle's own run of the same schedule, stored in
    tests/golden by make_anneal_record.py (which calls only the oracle): the
    realised schedule (stages, iterations of the fixed stages, the iteration
    count of the last stage within the stop-rule allowance of the reduced
    test) and the final potentials on the record's 256 sampled rows and
    columns after the gauge fix (f + c, g - c with c from the full means)."""
    with open(RECORD) as fh:
        rec = json.load(fh)
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(3, B=1)
    s = rec["schedule"]
    f, g, info = sot.sot_potentials_ex(dev(X), dev(Y), eps=s["eps_min"], eps_init=s["eps0"], eps_factor=s["factor"],
                                       iters_per_stage=s["iters_per_stage"], tol=s["tol"],
                                       max_iters=s["max_iters"], stats=True)
    gi = [int(v) for v in info["stage_iters"]][: info["stages_done"]]
    print(f"GPU: {info['stages_done']} stages, {info['iters_done']} iterations, converged {info['converged']}, "
          f"err {info['err'][0]:.4e}; oracle: {rec['stages_done']} stages, {rec['iters_done']} iterations, "
          f"converged {rec['converged']}, err {rec['err']:.4e}")
    assert info["stages_done"] == rec["stages_done"]
    assert gi[:-1] == rec["stage_iters"][:-1]  # the stages of fixed length
    ref = rec["iters_done"]
    assert abs(info["iters_done"] - ref) <= max(3, 0.02 * ref), (info["iters_done"], ref)
    fN, gN = host(f)[0], host(g)[0]
    c = rec["f_mean"] - float(np.mean(fN))
    rows, cols = np.array(rec["rows"]), np.array(rec["cols"])
    scale = max(rec["f_absmax"], rec["g_absmax"])
    ef = float(np.max(np.abs(fN[rows] + c - np.array(rec["f"])))) / scale
    eg = float(np.max(np.abs(gN[cols] - c - np.array(rec["g"])))) / scale
    print(f"sampled potentials (gauge-fixed): f {ef:.2e} g {eg:.2e}")
    assert ef < TOL and eg < TOL, (ef, eg)
