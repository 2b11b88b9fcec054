"""ctypes binding of the fp64 CPU oracle (``oracle.c``).

TEST INFRASTRUCTURE: only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline legs of ``bench.py`` import this module.  It shares no code with the
CUDA library.  Every array handed to the C code is float64; float32 inputs are
promoted exactly.

Each method works on one problem (X[n,d], Y[m,d], a[n], b[m]); the ``*_batch``
helpers loop over the leading batch axis.
"""
from __future__ import annotations

import contextlib
import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()

_dp = C.POINTER(C.c_double)
_ip = C.POINTER(C.c_int)


def build(mutant: int = 0, out_dir: str | None = None, force: bool = False) -> str:
    """Compile oracle.c into a shared library and return its path."""
    out_dir = out_dir or _BUILD
    os.makedirs(out_dir, exist_ok=True)
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    path = os.path.join(out_dir, name)
    with _lock:
        if force or not os.path.exists(path) or os.path.getmtime(path) < os.path.getmtime(_SRC):
            cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c99",
                   f"-DORC_MUTANT={int(mutant)}", _SRC, "-o", path + ".tmp", "-lm"]
            subprocess.run(cmd, check=True)
            os.replace(path + ".tmp", path)
    return path


def _d(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _ptr(x):
    return x.ctypes.data_as(_dp)


class Oracle:
    """fp64 Sinkhorn oracle loaded from a compiled ``oracle.c``."""

    def __init__(self, path: str | None = None, mutant: int = 0):
        self.path = path or build(mutant=mutant)
        self.lib = C.CDLL(self.path)
        L = self.lib
        L.orc_f_half.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, C.c_double, _dp]
        L.orc_g_half.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, _dp, C.c_double, _dp]
        L.orc_marginal_err.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, _dp, _dp, C.c_double]
        L.orc_marginal_err.restype = C.c_double
        L.orc_sinkhorn.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, C.c_int, _dp, _ip,
                                   _dp, _dp, C.c_int]
        L.orc_anneal_stages.argtypes = [C.c_double, C.c_double, C.c_double, _dp, C.c_int]
        L.orc_sinkhorn_anneal.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, C.c_double,
                                          C.c_double, C.c_double, C.c_int, C.c_double, C.c_int, C.c_int,
                                          _dp, _dp, C.c_int, _ip, C.c_int, _ip, _ip, _dp, _ip]
        L.orc_plan_apply.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, _dp, _dp, C.c_double,
                                     _dp, _dp, _dp, _dp]
        L.orc_objectives.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, _dp, _dp, C.c_double,
                                     _dp, _dp]
        L.orc_maxima.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, _dp, _dp, C.c_double,
                                 _dp, _dp]
        L.orc_coo.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, _dp, _dp, C.c_double,
                              C.c_double, C.c_int, C.c_double, C.c_longlong, _ip, _ip, _dp, _dp]
        L.orc_coo.restype = C.c_longlong
        L.orc_grad_support.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, C.c_longlong, _ip, _ip, _dp, _dp]
        L.orc_apml_coo.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, C.c_longlong, _ip, _ip,
                                   C.c_double, C.c_int, _dp, _dp]
        L.orc_num_threads.restype = C.c_int
        L.orc_set_num_threads.argtypes = [C.c_int]
        L.orc_mutant.restype = C.c_int
        L.orc_set_cost.argtypes = [C.c_int]
        L.orc_transport.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, _dp, _dp, C.c_double, _dp,
                                    C.c_int, C.c_int, _dp]
        L.orc_get_cost.restype = C.c_int
        L.orc_hvp.argtypes = [C.c_int, C.c_int, C.c_int, _dp, _dp, _dp, _dp, _dp, _dp, C.c_double, _dp, _dp, _dp,
                              _dp]

    # ---- plumbing -----------------------------------------------------
    @staticmethod
    def _prob(X, Y, a, b):
        X = _d(X)
        Y = _d(Y)
        if X.ndim == 1:
            X = X[:, None]
        if Y.ndim == 1:
            Y = Y[:, None]
        n, d = X.shape
        m, d2 = Y.shape
        if d != d2:
            raise ValueError("X and Y must have the same dimension")
        a = np.full(n, 1.0 / n) if a is None else _d(a)
        b = np.full(m, 1.0 / m) if b is None else _d(b)
        return X, Y, a, b, n, m, d

    @property
    def num_threads(self) -> int:
        return int(self.lib.orc_num_threads())

    def set_num_threads(self, t: int):
        self.lib.orc_set_num_threads(int(t))

    @property
    def mutant(self) -> int:
        return int(self.lib.orc_mutant())

    # ---- cost selection -------------------------------------------------
    COSTS = {"sqeuclidean": 0, "cosine": 1}

    @property
    def cost_kind(self) -> str:
        k = int(self.lib.orc_get_cost())
        return [name for name, v in self.COSTS.items() if v == k][0]

    @contextlib.contextmanager
    def cost(self, kind: str):
        """Select the cost for the calls inside the block ("sqeuclidean" or
        "cosine"); the previous selection is restored on exit."""
        prev = int(self.lib.orc_get_cost())
        self.lib.orc_set_cost(self.COSTS[kind])
        try:
            yield self
        finally:
            self.lib.orc_set_cost(prev)

    # ---- half steps ---------------------------------------------------
    def f_half(self, X, Y, b, g, eps):
        X, Y, _, b, n, m, d = self._prob(X, Y, None, b)
        g = _d(g)
        f = np.empty(n)
        rc = self.lib.orc_f_half(n, m, d, _ptr(X), _ptr(Y), _ptr(b), _ptr(g), float(eps), _ptr(f))
        if rc:
            raise RuntimeError(f"orc_f_half failed ({rc})")
        return f

    def g_half(self, X, Y, a, f, eps):
        X, Y, a, b, n, m, d = self._prob(X, Y, a, None)
        f = _d(f)
        g = np.empty(m)
        rc = self.lib.orc_g_half(n, m, d, _ptr(X), _ptr(Y), _ptr(a), _ptr(b), _ptr(f), float(eps), _ptr(g))
        if rc:
            raise RuntimeError(f"orc_g_half failed ({rc})")
        return g

    # ---- solves -------------------------------------------------------
    def sinkhorn(self, X, Y, a, b, eps_list, iters_list, f0=None, g0=None):
        """Fixed schedule: stage k runs iters_list[k] iterations at eps_list[k]."""
        X, Y, a, b, n, m, d = self._prob(X, Y, a, b)
        eps_list = np.ascontiguousarray(np.atleast_1d(eps_list), dtype=np.float64)
        iters = np.ascontiguousarray(np.atleast_1d(iters_list), dtype=np.int32)
        if eps_list.shape != iters.shape:
            raise ValueError("eps_list and iters_list differ in length")
        warm = f0 is not None or g0 is not None
        f = _d(np.zeros(n) if f0 is None else f0).copy()
        g = _d(np.zeros(m) if g0 is None else g0).copy()
        rc = self.lib.orc_sinkhorn(n, m, d, _ptr(X), _ptr(Y), _ptr(a), _ptr(b), len(iters), _ptr(eps_list),
                                   iters.ctypes.data_as(_ip), _ptr(f), _ptr(g), int(warm))
        if rc:
            raise RuntimeError(f"orc_sinkhorn failed ({rc})")
        return f, g

    def anneal_stages(self, eps0, factor, eps_min):
        k = self.lib.orc_anneal_stages(float(eps0), float(factor), float(eps_min), None, 0)
        if k <= 0:
            raise ValueError("bad annealing schedule")
        out = np.empty(k)
        self.lib.orc_anneal_stages(float(eps0), float(factor), float(eps_min), _ptr(out), k)
        return out

    def sinkhorn_anneal(self, X, Y, a, b, eps0, factor, eps_min, iters_per_stage, tol, max_iters,
                        early_exit=False, f0=None, g0=None):
        """Annealed solve with the marginal-error stop test (see oracle.c)."""
        X, Y, a, b, n, m, d = self._prob(X, Y, a, b)
        K = len(self.anneal_stages(eps0, factor, eps_min))
        warm = f0 is not None or g0 is not None
        f = _d(np.zeros(n) if f0 is None else f0).copy()
        g = _d(np.zeros(m) if g0 is None else g0).copy()
        st = np.zeros(K, dtype=np.int32)
        ns, it, conv = C.c_int(0), C.c_int(0), C.c_int(0)
        err = C.c_double(0)
        rc = self.lib.orc_sinkhorn_anneal(n, m, d, _ptr(X), _ptr(Y), _ptr(a), _ptr(b), float(eps0), float(factor),
                                          float(eps_min), int(iters_per_stage), float(tol), int(max_iters),
                                          int(bool(early_exit)), _ptr(f), _ptr(g), int(warm),
                                          st.ctypes.data_as(_ip), K, C.byref(ns), C.byref(it), C.byref(err),
                                          C.byref(conv))
        if rc:
            raise RuntimeError(f"orc_sinkhorn_anneal failed ({rc})")
        return dict(f=f, g=g, stage_iters=st[: ns.value].copy(), stages_done=ns.value, iters_done=it.value,
                    err=err.value, converged=bool(conv.value))

    # ---- outputs ------------------------------------------------------
    def marginal_err(self, X, Y, a, b, f, g, eps):
        X, Y, a, b, n, m, d = self._prob(X, Y, a, b)
        f, g = _d(f), _d(g)
        return float(self.lib.orc_marginal_err(n, m, d, _ptr(X), _ptr(Y), _ptr(a), _ptr(b), _ptr(f), _ptr(g),
                                               float(eps)))

    def plan_apply(self, X, Y, a, b, f, g, eps):
        """Returns dict(cost, grad[n,d], rowsum[n], colsum[m])."""
        X, Y, a, b, n, m, d = self._prob(X, Y, a, b)
        f, g = _d(f), _d(g)
        cost = C.c_double(0)
        grad = np.empty((n, d))
        r = np.empty(n)
        c = np.empty(m)
        rc = self.lib.orc_plan_apply(n, m, d, _ptr(X), _ptr(Y), _ptr(a), _ptr(b), _ptr(f), _ptr(g), float(eps),
                                     C.byref(cost), _ptr(grad), _ptr(r), _ptr(c))
        if rc:
            raise RuntimeError(f"orc_plan_apply failed ({rc})")
        return dict(cost=cost.value, grad=grad, rowsum=r, colsum=c)

    def transport(self, X, Y, a, b, f, g, eps, V, side=0):
        """Transport-matrix product: side 0 -> P V (V is m x c), side 1 -> P^T V
        (V is n x c).  A 1-D V gives a 1-D result."""
        X, Y, a, b, n, m, d = self._prob(X, Y, a, b)
        V = _d(V)
        vec = V.ndim == 1
        if vec:
            V = V[:, None]
        if V.shape[0] != (m if side == 0 else n):
            raise ValueError("V has the wrong number of rows for this side")
        c = V.shape[1]
        f, g = _d(f), _d(g)
        out = np.zeros(((n if side == 0 else m), c))
        rc = self.lib.orc_transport(n, m, d, _ptr(X), _ptr(Y), _ptr(a), _ptr(b), _ptr(f), _ptr(g),
                                    float(eps), _ptr(V), c, int(side), _ptr(out))
        if rc != 0:
            raise ValueError("orc_transport failed")
        return out[:, 0] if vec else out

    def hvp(self, X, Y, a, b, f, g, eps, V, derivs=False):
        """Hessian-vector product of the entropic OT loss with respect to X at
        the potentials (f, g), applied to V [n, d] (see orc_hvp).  With
        derivs=True also returns the potentials' first-order changes (fd, gd)."""
        X, Y, a, b, n, m, d = self._prob(X, Y, a, b)
        V = _d(V).reshape(n, d)
        f, g = _d(f), _d(g)
        out, fd, gd = np.empty((n, d)), np.empty(n), np.empty(m)
        rc = self.lib.orc_hvp(n, m, d, _ptr(X), _ptr(Y), _ptr(a), _ptr(b), _ptr(f), _ptr(g), float(eps), _ptr(V),
                              _ptr(out), _ptr(fd), _ptr(gd))
        if rc != 0:
            raise ValueError(f"orc_hvp failed ({rc})")
        return (out, fd, gd) if derivs else out

    def objectives(self, X, Y, a, b, f, g, eps):
        X, Y, a, b, n, m, d = self._prob(X, Y, a, b)
        f, g = _d(f), _d(g)
        du, pr = C.c_double(0), C.c_double(0)
        self.lib.orc_objectives(n, m, d, _ptr(X), _ptr(Y), _ptr(a), _ptr(b), _ptr(f), _ptr(g), float(eps),
                                C.byref(du), C.byref(pr))
        return du.value, pr.value

    def maxima(self, X, Y, a, b, f, g, eps):
        X, Y, a, b, n, m, d = self._prob(X, Y, a, b)
        f, g = _d(f), _d(g)
        Mr, Mc = np.empty(n), np.empty(m)
        self.lib.orc_maxima(n, m, d, _ptr(X), _ptr(Y), _ptr(a), _ptr(b), _ptr(f), _ptr(g), float(eps),
                            _ptr(Mr), _ptr(Mc))
        return Mr, Mc

    def coo(self, X, Y, a, b, f, g, eps, tau, dirs=3, band=0.0):
        """Pairs with margin >= -band, row-major: dict(rows, cols, vals, margins)."""
        X, Y, a, b, n, m, d = self._prob(X, Y, a, b)
        f, g = _d(f), _d(g)
        args = (n, m, d, _ptr(X), _ptr(Y), _ptr(a), _ptr(b), _ptr(f), _ptr(g), float(eps), float(tau),
                int(dirs), float(band))
        cnt = self.lib.orc_coo(*args, 0, None, None, None, None)
        if cnt < 0:
            raise ValueError(f"orc_coo failed ({cnt})")
        rows = np.empty(cnt, dtype=np.int32)
        cols = np.empty(cnt, dtype=np.int32)
        vals = np.empty(cnt)
        mar = np.empty(cnt)
        cnt2 = self.lib.orc_coo(*args, cnt, rows.ctypes.data_as(_ip), cols.ctypes.data_as(_ip), _ptr(vals),
                                _ptr(mar))
        assert cnt2 == cnt
        return dict(rows=rows, cols=cols, vals=vals, margins=mar)

    def grad_support(self, X, Y, rows, cols, vals):
        X, Y, _, _, n, m, d = self._prob(X, Y, None, None)
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        cols = np.ascontiguousarray(cols, dtype=np.int32)
        vals = _d(vals)
        grad = np.empty((n, d))
        rc = self.lib.orc_grad_support(n, m, d, _ptr(X), _ptr(Y), len(rows), rows.ctypes.data_as(_ip),
                                       cols.ctypes.data_as(_ip), _ptr(vals), _ptr(grad))
        if rc:
            raise ValueError("orc_grad_support: index out of range")
        return grad

    def apml_coo(self, X, Y, a, b, rows, cols, T, iters):
        """Sparse APML on a row-major support: (P values on the support, loss)."""
        X, Y, a, b, n, m, d = self._prob(X, Y, a, b)
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        cols = np.ascontiguousarray(cols, dtype=np.int32)
        vals = np.empty(len(rows))
        loss = C.c_double(0)
        rc = self.lib.orc_apml_coo(n, m, d, _ptr(X), _ptr(Y), _ptr(a), _ptr(b), len(rows),
                                   rows.ctypes.data_as(_ip), cols.ctypes.data_as(_ip), float(T), int(iters),
                                   _ptr(vals), C.byref(loss))
        if rc:
            raise ValueError(f"orc_apml_coo failed ({rc})")
        return vals, loss.value

    # ---- batch helpers -----------------------------------------------
    def sinkhorn_batch(self, X, Y, a, b, eps, iters, clouds=None):
        idx = range(X.shape[0]) if clouds is None else clouds
        out = [self.sinkhorn(X[k], Y[k], None if a is None else a[k], None if b is None else b[k],
                             [eps], [iters]) for k in idx]
        return np.stack([o[0] for o in out]), np.stack([o[1] for o in out])


_default = None


def get() -> Oracle:
    """The shared (non-mutant) oracle instance."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default
