"""Device memory of a call stays linear in the cloud sizes ("FlashSinkhorn",
Methodologie 3 and its results: working memory O((n + m) d), the n x m plan is
never stored).

Free device memory is read before and after the calls, with every input and
output allocated beforehand and a small warm-up call first (so kernel code
loaded on first use is not counted).  The library's scratch pool keeps up to
2 GiB of freed scratch, so what the calls took is still held when the second
reading is taken; the bound below (a tenth of the dense fp32 plan) sits under
that 2 GiB, so a larger peak could not hide behind memory handed back."""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sot():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sinkhorn_point_cloud_gb300 as s
    from sinkhorn_point_cloud_gb300 import build
    build.build()
    return s


def _used_by(sot, wid, iters):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    w = dg.WORKLOADS[wid]
    B, n, m, d, eps = w["B"], w["n"], w["m"], w["d"], w["eps"]
    X, Y, a, b = dg.make_batch(wid, B=B)
    weighted = w["kind"] == "gauss"
    Xd, Yd = torch.from_numpy(X).cuda(), torch.from_numpy(Y).cuda()
    ad, bd = (torch.from_numpy(a).cuda(), torch.from_numpy(b).cuda()) if weighted else (None, None)
    f, g = torch.empty(B, n, device="cuda"), torch.empty(B, m, device="cuda")
    cost, grad = torch.empty(B, device="cuda"), torch.empty(B, n, d, device="cuda")
    # warm-up on a slice of the same workload: the same kernels, loaded once
    k = min(n, m, 1000)
    Xs, Ys = Xd[:1, :k].contiguous(), Yd[:1, :k].contiguous()
    fs, gs = torch.empty(1, k, device="cuda"), torch.empty(1, k, device="cuda")
    sot.sot_potentials(Xs, Ys, eps=eps, iters=3, f=fs, g=gs)
    sot.sot_plan_apply(Xs, Ys, None, None, fs, gs, eps)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    sot.sot_potentials(Xd, Yd, ad, bd, eps=eps, iters=iters, f=f, g=g)
    sot.sot_plan_apply(Xd, Yd, ad, bd, f, g, eps, cost=cost, grad=grad)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert np.isfinite(cost.cpu().numpy()).all()
    return free0 - free1, 4.0 * B * n * m


@pytest.mark.parametrize("wid,iters", [(4, 10), (5, 20)])
def test_call_memory_is_far_below_the_dense_plan(sot, wid, iters):
    used, dense = _used_by(sot, wid, iters)
    print(f"workload {wid}: {used / 2**20:.1f} MiB held after the calls; a dense fp32 plan is {dense / 2**20:.0f} MiB")
    assert used < dense / 10, (used, dense)
