"""Cluster-resident iterations of the point path (d <= 3, clouds that fit in
shared memory) vs the fp64 oracle and vs the streaming half-steps.

Sizes cover odd and unequal cloud sizes (a padding column in the pair
layout), clusters whose last CTAs own fewer rows, several clouds per launch,
d = 1, 2, 3, and more clouds than fit at the largest cluster size.  The
solver takes the cluster path only where its cost model expects a gain (small
problems); the 32-cloud workload at full size streams."""
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


def solve(sot, X, Y, eps, iters, flags):
    sot.sot_profile_read_kinds()
    sot.sot_profile_enable(True)
    f, g = sot.sot_potentials_ex(dev(X), dev(Y), None, None, eps=eps, iters_per_stage=iters, max_iters=iters,
                                 flags=flags)
    kinds = sot.sot_profile_read_kinds()
    sot.sot_profile_enable(False)
    return host(f), host(g), kinds


@pytest.mark.parametrize("w,B,n,m,d,eps,iters", [
    (1, 1, 256, 256, 3, 0.01, 100),   # the 256-point workload, whole
    (1, 3, 301, 257, 3, 0.02, 60),    # odd sizes, three clouds
    (2, 2, 500, 377, 3, 0.01, 80),    # sphere + rotation, unequal sizes
    (1, 2, 95, 130, 2, 0.05, 50),     # d = 2, fewer rows than cluster threads
    (1, 1, 9, 14, 1, 0.1, 40),        # d = 1, CTAs without rows
])
def test_cluster_matches_oracle(sot, orc, w, B, n, m, d, eps, iters):
    """Every case here is small enough that the solver takes the cluster path."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(w, B=B, n=n, m=m, d=d)
    f, g, kinds = solve(sot, X, Y, eps, iters, 0)
    assert kinds["cluster"][0] == 2 * (iters - 1), kinds  # the cold first iteration streams
    sols = [orc.sinkhorn(X[k], Y[k], a[k], b[k], [eps], [iters]) for k in range(B)]
    fr, gr = np.stack([s[0] for s in sols]), np.stack([s[1] for s in sols])
    ef, eg = potentials_error(f, g, fr, gr)
    print(f"cluster vs oracle: f {ef:.2e} g {eg:.2e}")
    assert ef < TOL and eg < TOL, (ef, eg)


def test_cluster_agrees_with_streaming(sot):
    """Clouds of the 32-cloud recipe (two of n = m = 512): cluster-resident and
    streaming iterations give the same potentials to well below the parity
    tolerance, and the plan applied to them gives the same cost and, within the
    parity tolerance, the same gradient."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(2, B=2, n=512)
    eps, iters = 0.01, 200
    fc, gc, kc = solve(sot, X, Y, eps, iters, 0)
    fs, gs, ks = solve(sot, X, Y, eps, iters, sot.SOT_NO_CLUSTER)
    assert kc["cluster"][0] == 2 * (iters - 1) and ks["cluster"][0] == 0, (kc, ks)
    ef, eg = potentials_error(fc, gc, fs, gs)
    assert ef < 2e-5 and eg < 2e-5, (ef, eg)
    Xd, Yd = dev(X), dev(Y)
    c1, g1 = sot.sot_cost_grad(Xd, Yd, None, None, dev(fc.astype(np.float32)), dev(gc.astype(np.float32)), eps)
    c2, g2 = sot.sot_cost_grad(Xd, Yd, None, None, dev(fs.astype(np.float32)), dev(gs.astype(np.float32)), eps)
    # (the gradient amplifies potential differences by ~1/eps)
    assert normwise(host(c1), host(c2)) < 2e-5 and normwise(host(g1), host(g2)) < TOL


def test_cluster_many_clouds(sot, orc):
    """More clouds than fit at 8 CTAs each on the device (B = 40): the cluster
    size drops to keep one wave; sampled clouds against the oracle."""
    from sinkhorn_point_cloud_gb300 import datagen as dg
    B, n, eps, iters = 40, 200, 0.02, 30
    X, Y, a, b = dg.make_batch(2, B=B, n=n)
    f, g, kinds = solve(sot, X, Y, eps, iters, 0)
    assert kinds["cluster"][0] == 2 * (iters - 1), kinds
    sel = [0, 17, 39]
    sols = [orc.sinkhorn(X[k], Y[k], a[k], b[k], [eps], [iters]) for k in sel]
    fr, gr = np.stack([s[0] for s in sols]), np.stack([s[1] for s in sols])
    ef, eg = potentials_error(f[sel], g[sel], fr, gr)
    assert ef < TOL and eg < TOL, (ef, eg)
