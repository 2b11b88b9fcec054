"""sot_potentials_noalloc: the potentials solve for callers that cannot
allocate device memory on the call path (for example when another
framework's caching allocator has reserved all device memory up front, or in
latency-critical loops where an allocator call and the synchronisation it
can trigger are not allowed).  Its scratch is the library's static device
array, so consecutive calls reuse the same memory; each call must still give
the same potentials as sot_potentials.

This file is collected last so that a failure here does not hide the others.
"""
import ctypes as C

import numpy as np
import pytest

from gpu_util import TOL, dev, host, potentials_error


def _problem(seed_cloud, n, m):
    from sinkhorn_point_cloud_gb300 import datagen as dg
    return dg.make_batch(2, B=3, n=n, m=m, clouds=range(seed_cloud, seed_cloud + 3))


@pytest.mark.gpu
def test_noalloc_matches_sot_potentials_on_two_calls_in_a_row():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sinkhorn_point_cloud_gb300 as sot
    from sinkhorn_point_cloud_gb300 import build
    build.build()
    eps, iters = 0.01, 60
    # two different problems, one call each, back to back: the second call must
    # not see anything the first one left in the shared scratch
    for seed, (n, m) in ((0, (700, 555)), (5, (513, 640))):
        X, Y, a, b = _problem(seed, n, m)
        Xd, Yd = dev(X), dev(Y)
        f_ref, g_ref = sot.sot_potentials(Xd, Yd, eps=eps, iters=iters)
        f = torch.empty(3, n, device="cuda")
        g = torch.empty(3, m, device="cuda")
        sot.sot_potentials_noalloc(Xd, Yd, eps=eps, iters=iters, f=f, g=g)
        torch.cuda.synchronize()
        ef, eg = potentials_error(host(f), host(g), host(f_ref), host(g_ref))
        assert ef < TOL and eg < TOL, (n, m, ef, eg)


def test_noalloc_rejects_problems_beyond_the_static_scratch():
    """Checked on the host before anything is launched (no GPU needed)."""
    from sinkhorn_point_cloud_gb300 import binding, build
    build.build()
    L = binding.load()
    p = C.c_void_p(16)  # never dereferenced: the size check fails first
    rc = L.sot_potentials_noalloc(p, p, None, None, 64, 65536, 65536, 3, 0.01, 10, p, p, None)
    assert rc == binding.SOT_ERR_INVALID_ARG
    assert b"static area holds" in L.sot_last_error()
    rc = L.sot_potentials_noalloc(p, p, None, None, 1, 100, 100, 8, 0.01, 10, p, p, None)
    assert rc == binding.SOT_ERR_UNSUPPORTED
