"""Build and call the fp32 COO replica (``coo_replica.c``), a test checker.

It re-decides libsot's thresholded COO support from the fp32 operands that
``sot_plan_coo_operands`` reports.  It is not the oracle and shares no code
with it or with the library.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "coo_replica.c")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libcooreplica.so")

_lib = None


def build() -> str:
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", SRC, "-o", LIB + ".tmp", "-lm"]
    subprocess.run(cmd, check=True, capture_output=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


def _load():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        P, i, f, ll = C.c_void_p, C.c_int, C.c_float, C.c_longlong
        L.coo_replica.argtypes = [i, i, i, P, P, P, P, P, P, f, f, i, P, P, ll, P, P]
        L.coo_replica.restype = ll
        _lib = L
    return _lib


def _f32(a):
    return np.ascontiguousarray(a, dtype=np.float32)


def replica(xc, lwx, Lx, yc, lwy, Ly, kappa, log2tau, dirs):
    """One cloud: returns dict(rows, cols, Mr, Mc) from the replica."""
    L = _load()
    xc, lwx, Lx, yc, lwy, Ly = map(_f32, (xc, lwx, Lx, yc, lwy, Ly))
    n, d = xc.shape
    m = yc.shape[0]
    Mr = np.empty(n, np.float32)
    Mc = np.empty(m, np.float32)
    ptr = lambda a: a.ctypes.data_as(C.c_void_p)
    args = [n, m, d, ptr(xc), ptr(lwx), ptr(Lx), ptr(yc), ptr(lwy), ptr(Ly), C.c_float(kappa), C.c_float(log2tau),
            int(dirs), ptr(Mr), ptr(Mc)]
    nnz = L.coo_replica(*args, 0, None, None)
    if nnz < 0:
        raise RuntimeError(f"coo_replica failed ({nnz})")
    rows = np.empty(max(nnz, 1), np.int32)
    cols = np.empty(max(nnz, 1), np.int32)
    got = L.coo_replica(*args, nnz, ptr(rows), ptr(cols))
    assert got == nnz
    return dict(rows=rows[:nnz], cols=cols[:nnz], Mr=Mr, Mc=Mc)
