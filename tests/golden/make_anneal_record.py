"""Writes anneal_gmm8_n16384_cloud0.json: the fp64 oracle's annealed solve of
cloud 0 of the 4-cloud Gaussian-mixture workload at full size (n = m = 16384,
d = 3; eps 1 -> 1e-3 by x0.9 per stage, 20 iterations per stage, stop at a
marginal L1 error below 1e-4 at the final eps, at most 5000 iterations).

The record holds the realised schedule (per-stage iterations, whether the stop
test passed, the final marginal error) and the final potentials on 256 seeded
sampled rows and columns, for tests/test_gpu_anneal.py.  It calls only the
oracle and the seeded input generator; it takes about an hour on 8 cores.

    python tests/golden/make_anneal_record.py
"""
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


def main():
    orc = O.get()
    X, Y, a, b = dg.make_batch(3, B=1)
    t0 = time.time()
    out = orc.sinkhorn_anneal(X[0], Y[0], None, None, **SCHEDULE)
    secs = time.time() - t0
    rng = np.random.default_rng(20261203)
    rows = np.sort(rng.choice(X.shape[1], 256, replace=False))
    cols = np.sort(rng.choice(Y.shape[1], 256, replace=False))
    rec = dict(
        workload="gmm8_B4_n16384_d3_annealed", cloud=0, n=int(X.shape[1]), m=int(Y.shape[1]), schedule=SCHEDULE,
        stages_done=int(out["stages_done"]), stage_iters=[int(v) for v in out["stage_iters"]],
        iters_done=int(out["iters_done"]), converged=bool(out["converged"]), err=float(out["err"]),
        rows=rows.tolist(), f=[float(v) for v in out["f"][rows]],
        cols=cols.tolist(), g=[float(v) for v in out["g"][cols]],
        f_mean=float(np.mean(out["f"])), g_mean=float(np.mean(out["g"])),
        f_absmax=float(np.max(np.abs(out["f"]))), g_absmax=float(np.max(np.abs(out["g"]))),
        oracle_threads=int(orc.num_threads()) if hasattr(orc, "num_threads") else None, seconds=round(secs, 1))
    with open(OUT, "w") as fh:
        json.dump(rec, fh, indent=1)
    print(f"{OUT}: {rec['iters_done']} iterations, converged {rec['converged']}, err {rec['err']:.4e}, {secs:.0f} s")


if __name__ == "__main__":
    main()
