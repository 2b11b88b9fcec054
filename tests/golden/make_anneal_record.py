"""Writes anneal_gmm8_n16384_cloud0.json: the fp64 oracle's annealed solve of
cloud 0 of the 4-cloud Gaussian-mixture workload at full size (n = m = 16384,
d = 3; eps 1 -> 1e-3 by x0.9 per stage, 20 iterations per stage, stop at a
marginal L1 error below 1e-4 at the final eps, at most 5000 iterations).

The record holds the realised schedule (per-stage iterations, whether the stop
test passed, the final marginal error) and the final potentials on 256 seeded
sampled rows and columns, for tests/test_gpu_anneal.py.  It calls only the
oracle and the seeded input generator.

The solve takes about four hours on 8 x86 cores (about one on 16 Arm cores:
the last stage's marginal-error test after every iteration costs more than the
iteration), so it runs in pieces, each a call of the
oracle that continues from the previous piece's potentials: the stages of
fixed length one at a time (the oracle's fixed-schedule solve, one stage), then
the last stage in chunks of iterations (the oracle's annealed solve on that one
stage, whose stop test runs after every iteration as in the last stage of the
whole schedule, with the iteration cap that is left).  The pieces compose to the
oracle's single annealed call exactly (tests/test_oracle_pins.py checks that on
a small problem).  After every piece the potentials and counters go to a
checkpoint file, so an interrupted run resumes where it stopped:

    python tests/golden/make_anneal_record.py [--checkpoint PATH] [--chunk ITERS]
"""
import argparse
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

from oracle import oracle as O  # noqa: E402
from sinkhorn_point_cloud_gb300 import datagen as dg  # noqa: E402

OUT = os.path.join(HERE, "anneal_gmm8_n16384_cloud0.json")
SCHEDULE = dict(eps0=1.0, factor=0.9, eps_min=1e-3, iters_per_stage=20, tol=1e-4, max_iters=5000)


def anneal_in_pieces(orc, X, Y, schedule, state=None, chunk=100, save=None):
    """The annealed solve of `schedule` (uniform weights) as a sequence of
    oracle calls.  `state` (a dict from a previous, interrupted run, or None)
    holds f, g, the per-stage iterations done, the total, err and whether the
    stop test passed; `save(state)` is called after every piece.  Returns the
    final state: the same quantities as the oracle's single annealed call."""
    eps = orc.anneal_stages(schedule["eps0"], schedule["factor"], schedule["eps_min"])
    K, per, cap = len(eps), int(schedule["iters_per_stage"]), int(schedule["max_iters"])
    if state is None:
        state = dict(f=np.zeros(X.shape[0]), g=np.zeros(Y.shape[0]), stage_iters=[], total=0, err=float("nan"),
                     converged=False, seconds=0.0)
    while True:
        k = len(state["stage_iters"]) - (1 if state.get("open") else 0)
        if state["converged"] or state["total"] >= cap or k >= K:
            break
        t0 = time.time()
        if k < K - 1:
            # a stage of fixed length: no stop test
            it = min(per, cap - state["total"])
            f, g = orc.sinkhorn(X, Y, None, None, [eps[k]], [it], f0=state["f"], g0=state["g"])
            state["stage_iters"].append(it)
            state["total"] += it
        else:
            # the last stage: tested after every iteration, up to the cap
            if not state.get("open"):
                state["stage_iters"].append(0)
                state["open"] = True
            it = min(chunk, cap - state["total"])
            out = orc.sinkhorn_anneal(X, Y, None, None, eps[k], schedule["factor"], eps[k], per,
                                      schedule["tol"], it, f0=state["f"], g0=state["g"])
            f, g = out["f"], out["g"]
            state["stage_iters"][-1] += out["iters_done"]
            state["total"] += out["iters_done"]
            state["err"] = out["err"]
            state["converged"] = out["converged"]
        state["f"], state["g"] = f, g
        state["seconds"] += time.time() - t0
        if save:
            save(state)
    state["stages_done"] = len(state["stage_iters"])
    return state


def _load(path):
    if not path or not os.path.exists(path):
        return None
    z = np.load(path, allow_pickle=False)
    meta = json.loads(str(z["meta"]))
    return dict(f=z["f"], g=z["g"], **meta)


def _saver(path):
    def save(state):
        meta = {k: v for k, v in state.items() if k not in ("f", "g")}
        tmp = path + ".tmp.npz"
        np.savez(tmp, f=state["f"], g=state["g"], meta=json.dumps(meta))
        os.replace(tmp, path)
        print(f"  {state['total']} iterations, {len(state['stage_iters'])} stages, err {state['err']:.4e}, "
              f"{state['seconds']:.0f} s", flush=True)
    return save if path else None


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--checkpoint", default=os.path.join(HERE, "anneal_record_checkpoint.npz"))
    ap.add_argument("--chunk", type=int, default=100, help="iterations of the last stage per piece")
    args = ap.parse_args()
    orc = O.get()
    X, Y, a, b = dg.make_batch(3, B=1)
    out = anneal_in_pieces(orc, X[0], Y[0], SCHEDULE, state=_load(args.checkpoint), chunk=args.chunk,
                           save=_saver(args.checkpoint))
    rng = np.random.default_rng(20261203)
    rows = np.sort(rng.choice(X.shape[1], 256, replace=False))
    cols = np.sort(rng.choice(Y.shape[1], 256, replace=False))
    f, g = np.asarray(out["f"]), np.asarray(out["g"])
    rec = dict(
        workload="gmm8_B4_n16384_d3_annealed", cloud=0, n=int(X.shape[1]), m=int(Y.shape[1]), schedule=SCHEDULE,
        stages_done=int(out["stages_done"]), stage_iters=[int(v) for v in out["stage_iters"]],
        iters_done=int(out["total"]), converged=bool(out["converged"]), err=float(out["err"]),
        rows=rows.tolist(), f=[float(v) for v in f[rows]],
        cols=cols.tolist(), g=[float(v) for v in g[cols]],
        f_mean=float(np.mean(f)), g_mean=float(np.mean(g)),
        f_absmax=float(np.max(np.abs(f))), g_absmax=float(np.max(np.abs(g))),
        oracle_threads=int(orc.num_threads), seconds=round(float(out["seconds"]), 1))
    with open(OUT, "w") as fh:
        json.dump(rec, fh, indent=1)
    print(f"{OUT}: {rec['iters_done']} iterations, converged {rec['converged']}, err {rec['err']:.4e}, "
          f"{rec['seconds']:.0f} s")


if __name__ == "__main__":
    main()
