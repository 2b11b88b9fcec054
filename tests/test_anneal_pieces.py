"""The stored record of the full-size annealed solve is computed in pieces
(tests/golden/make_anneal_record.py): each fixed-length stage as a one-stage
fixed-schedule call, then the last stage in chunks, each an annealed call on
that single stage with the iteration cap left.  Here, on small problems, the
pieces must give exactly what the oracle's single annealed call gives: the
realised schedule, the stop decision, the marginal error and the potentials,
including runs interrupted and resumed from a checkpoint."""
import importlib.util
import os

import numpy as np
import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


def _script():
    spec = importlib.util.spec_from_file_location("make_anneal_record",
                                                  os.path.join(HERE, "golden", "make_anneal_record.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _single(orc, X, Y, s):
    return orc.sinkhorn_anneal(X, Y, None, None, s["eps0"], s["factor"], s["eps_min"], s["iters_per_stage"],
                               s["tol"], s["max_iters"])


@pytest.mark.parametrize("tol,max_iters", [
    (3e-3, 2000),   # the last stage stops on the test
    (1e-12, 260),   # the cap falls inside the last stage
    (1e-12, 53),    # the cap falls inside a stage of fixed length (11 of them, 55 iterations)
    (1e-12, 50),    # the cap falls on the end of a stage of fixed length
    (1e-12, 55),    # the cap falls on the end of the last stage of fixed length
])
def test_pieces_match_the_single_annealed_call(orc, tol, max_iters):
    mod = _script()
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, _, _ = dg.make_batch(3, B=1, n=140, m=130)
    X, Y = X[0], Y[0]
    s = dict(eps0=1.0, factor=0.7, eps_min=0.02, iters_per_stage=5, tol=tol, max_iters=max_iters)
    ref = _single(orc, X, Y, s)
    assert len(orc.anneal_stages(s["eps0"], s["factor"], s["eps_min"])) == 12
    got = mod.anneal_in_pieces(orc, X, Y, s, chunk=7)
    assert got["stages_done"] == ref["stages_done"]
    assert got["stage_iters"] == [int(v) for v in ref["stage_iters"]]
    assert got["total"] == ref["iters_done"]
    assert got["converged"] == ref["converged"]
    if np.isnan(ref["err"]):
        assert np.isnan(got["err"])
    else:
        assert got["err"] == ref["err"]
    assert np.array_equal(got["f"], ref["f"]) and np.array_equal(got["g"], ref["g"])
    if tol > 1e-6:
        assert ref["converged"] and ref["err"] < tol


def test_pieces_resume_from_a_checkpoint(orc, tmp_path):
    mod = _script()
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, _, _ = dg.make_batch(3, B=1, n=120, m=110)
    X, Y = X[0], Y[0]
    s = dict(eps0=1.0, factor=0.7, eps_min=0.02, iters_per_stage=5, tol=1e-12, max_iters=120)
    ref = _single(orc, X, Y, s)
    path = str(tmp_path / "ck.npz")
    save = mod._saver(path)
    calls = []

    def stop_after_four(state):
        save(state)
        calls.append(1)
        if len(calls) == 4 or len(calls) == 13:
            raise KeyboardInterrupt

    for _ in range(3):
        try:
            got = mod.anneal_in_pieces(orc, X, Y, s, state=mod._load(path), chunk=9, save=stop_after_four)
            break
        except KeyboardInterrupt:
            continue
    assert len(calls) > 13
    assert got["stage_iters"] == [int(v) for v in ref["stage_iters"]]
    assert got["total"] == ref["iters_done"]
    assert np.array_equal(got["f"], ref["f"]) and np.array_equal(got["g"], ref["g"])
