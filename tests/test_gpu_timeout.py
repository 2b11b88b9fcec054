"""Bounded device-side waits of the tensor-core kernels give up cleanly.

Every mbarrier wait in the tensor-core kernels has a time limit.  A kernel
whose wait runs out must wait for the bulk copies and MMAs it already issued,
free its TMEM, leave NaN in the rows it held and report SOT_ERR_TIMEOUT, and
the device must stay usable.  The failure is made by a testing hook
(sot_test_hold_tile): the producer withholds a column tile's copy, so the
waits on it run out after a 1 ms limit; nothing faults and nothing hangs.
"""
import numpy as np
import pytest

from gpu_util import TOL, dev, host, normwise, potentials_error

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

LIMIT_NS = 1_000_000  # 1 ms


@pytest.fixture(scope="module")
def sot():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sinkhorn_point_cloud_gb300 as s
    from sinkhorn_point_cloud_gb300 import build
    build.build()
    if s.sot_select_path(64, 0) != 2:
        pytest.skip("tensor-core path not built")
    return s


@pytest.fixture(scope="module")
def prob():
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=4096, m=4096, d=64)
    return dev(X), dev(Y), dev(a), dev(b)


@pytest.fixture(autouse=True)
def hook_off(sot):
    yield
    sot.sot_test_hold_tile(-1)


@pytest.mark.parametrize("tile,after", [(0, 0), (1, 0), (1, 2)],
                         ids=["first tile (nothing but the row tiles in flight)",
                              "second tile (MMAs of the first in flight)",
                              "screened half-step (after two full half-steps)"])
def test_timeout_reported_with_stats(sot, prob, tile, after):
    Xd, Yd, ad, bd = prob
    sot.sot_test_hold_tile(tile, after, LIMIT_NS)
    with pytest.raises(sot.SotError) as ei:
        sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=0.1, iters_per_stage=3, stats=True)
    assert ei.value.status == sot.SOT_ERR_TIMEOUT


def test_timeout_reported_asynchronously(sot, prob):
    Xd, Yd, ad, bd = prob
    sot.sot_async_status()  # clears what earlier calls left
    sot.sot_test_hold_tile(1, 2, LIMIT_NS)
    f, g = sot.sot_potentials(Xd, Yd, ad, bd, eps=0.1, iters=3)
    with pytest.raises(sot.SotError) as ei:
        sot.sot_async_status()
    assert ei.value.status == sot.SOT_ERR_TIMEOUT
    assert torch.isnan(f).any() and torch.isnan(g).any()
    sot.sot_async_status()  # cleared by the previous read


def test_plan_application_timeout(sot, prob):
    Xd, Yd, ad, bd = prob
    f, g = sot.sot_potentials(Xd, Yd, ad, bd, eps=0.1, iters=3)
    sot.sot_async_status()
    sot.sot_test_hold_tile(1, 0, LIMIT_NS)
    c, gr, _ = sot.sot_plan_apply(Xd, Yd, ad, bd, f, g, 0.1)
    with pytest.raises(sot.SotError) as ei:
        sot.sot_async_status()
    assert ei.value.status == sot.SOT_ERR_TIMEOUT
    assert torch.isnan(gr).any()


def test_device_usable_after_timeouts(sot, orc, prob):
    """After every case above, on the same device: a normal solve reports no
    timeout and matches the oracle."""
    Xd, Yd, ad, bd = prob
    sot.sot_test_hold_tile(0, 0, LIMIT_NS)
    with pytest.raises(sot.SotError):
        sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=0.1, iters_per_stage=2, stats=True)
    sot.sot_test_hold_tile(-1)
    sot.sot_async_status()
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=600, m=520, d=64)
    eps, iters = 0.1, 50
    f, g, st = sot.sot_potentials_ex(dev(X), dev(Y), dev(a), dev(b), eps=eps, iters_per_stage=iters,
                                     stats=True)
    c, gr, _ = sot.sot_plan_apply(dev(X), dev(Y), dev(a), dev(b), f, g, eps)
    sot.sot_async_status()
    fr, gref = orc.sinkhorn(X[0], Y[0], a[0], b[0], [eps], [iters])
    ef, eg = potentials_error(host(f), host(g), fr[None], gref[None])
    # the plan application, on the GPU's own potentials (its sensitivity to the
    # potentials is 1/eps: compared on the same ones)
    out = orc.plan_apply(X[0], Y[0], a[0], b[0], host(f)[0], host(g)[0], eps)
    egr = normwise(host(gr)[0], out["grad"])
    assert max(ef, eg, egr) < TOL, (ef, eg, egr)


@pytest.fixture(scope="module")
def prob_wide():
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=4096, m=4096, d=128)
    return dev(X), dev(Y), dev(a), dev(b)


@pytest.mark.parametrize("tile,after", [(1, 0), (1, 2)],
                         ids=["sliced full half-step", "sliced screened half-step"])
def test_timeout_sliced_kernels(sot, orc, prob_wide, tile, after):
    """d = 128: the kernels that stream K slices (the full and the screened
    half-step) give up the same way; a plan application with a withheld tile
    reports it asynchronously; a normal solve on the same device afterwards
    matches the oracle."""
    Xd, Yd, ad, bd = prob_wide
    sot.sot_test_hold_tile(tile, after, LIMIT_NS)
    with pytest.raises(sot.SotError) as ei:
        sot.sot_potentials_ex(Xd, Yd, ad, bd, eps=0.2, iters_per_stage=3, stats=True)
    assert ei.value.status == sot.SOT_ERR_TIMEOUT
    sot.sot_test_hold_tile(-1)
    f, g = sot.sot_potentials(Xd, Yd, ad, bd, eps=0.2, iters=3)
    sot.sot_async_status()
    sot.sot_test_hold_tile(1, 0, LIMIT_NS)
    c, gr, _ = sot.sot_plan_apply(Xd, Yd, ad, bd, f, g, 0.2)
    with pytest.raises(sot.SotError) as ei:
        sot.sot_async_status()
    assert ei.value.status == sot.SOT_ERR_TIMEOUT
    assert torch.isnan(gr).any()
    sot.sot_test_hold_tile(-1)
    from sinkhorn_point_cloud_gb300 import datagen as dg
    X, Y, a, b = dg.make_batch(4, B=1, n=400, m=360, d=128)
    f, g = sot.sot_potentials(dev(X), dev(Y), dev(a), dev(b), eps=0.2, iters=30)
    sot.sot_async_status()
    fr, gref = orc.sinkhorn(X[0], Y[0], a[0], b[0], [0.2], [30])
    ef, eg = potentials_error(host(f), host(g), fr[None], gref[None])
    assert max(ef, eg) < TOL, (ef, eg)
