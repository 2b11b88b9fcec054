"""Thin ctypes binding of libsot (include/sot.h), same names as the C ABI.

Only argument marshalling lives here: every step of the computation runs in
the CUDA kernels of libsot.  Tensors must be float32, contiguous and on the
current CUDA device; the calls are stream-ordered on
``torch.cuda.current_stream()`` unless a stream is given.  Outputs are
allocated with torch when not supplied (plain device memory, no compute).
A missing or unloadable libsot raises at once: there is no CPU fallback.
"""
from __future__ import annotations

import ctypes as C
import os
import re

import torch

from . import build as _build

SOT_OK = 0
SOT_ERR_INVALID_ARG = -1
SOT_ERR_NONFINITE = -2
SOT_ERR_CAPACITY = -3
SOT_ERR_TIMEOUT = -4
SOT_ERR_CUDA = -5
SOT_ERR_UNSUPPORTED = -6
SOT_ERR_NOMEM = -7

SOT_PREC_AUTO = 0
SOT_PREC_FP32 = 1
SOT_PREC_F16X3 = 2
SOT_WARM_START = 1 << 4
SOT_STAGE_EARLY_EXIT = 1 << 5
SOT_TC_NO_SCREEN = 1 << 6
SOT_NO_CLUSTER = 1 << 7
SOT_COST_COSINE = 1 << 8

HEADER = os.path.join(_build.ROOT, "include", "sot.h")


class SotError(RuntimeError):
    def __init__(self, status: int, func: str, detail: str):
        super().__init__(f"{func}: {detail} (status {status})")
        self.status = status


class sot_schedule(C.Structure):
    _fields_ = [("eps", C.c_float), ("eps_init", C.c_float), ("eps_factor", C.c_float),
                ("iters_per_stage", C.c_int), ("max_iters", C.c_int), ("tol", C.c_float), ("flags", C.c_int)]


class sot_stats(C.Structure):
    _fields_ = [("iters_done", C.c_int), ("stages_done", C.c_int), ("converged", C.c_int), ("final_eps", C.c_float),
                ("err_host", C.POINTER(C.c_float)), ("stage_iters_host", C.POINTER(C.c_int)),
                ("stage_iters_cap", C.c_int)]


_lib = None
_fp = C.c_void_p


def declared_functions() -> list[str]:
    """Names of the functions declared in include/sot.h."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(sot_[a-z_0-9]+)\s*\(", txt)))


def load(path: str | None = None):
    """Load libsot.so (built in-tree by ``build.build()``); raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _build.LIB
    if not os.path.exists(p):
        raise RuntimeError(f"libsot.so not found at {p}: run sinkhorn_point_cloud_gb300.build.build()")
    L = C.CDLL(p)
    P = _fp
    i, f, ll = C.c_int, C.c_float, C.c_longlong
    sig = {
        "sot_potentials": [P, P, P, P, i, i, i, i, f, i, P, P, P],
        "sot_potentials_ex": [P, P, P, P, i, i, i, i, C.POINTER(sot_schedule), P, P, C.POINTER(sot_stats), P],
        "sot_plan_apply": [P, P, P, P, i, i, i, i, P, P, f, P, P, P, i, P],
        "sot_cost": [P, P, P, P, i, i, i, i, P, P, f, P, P],
        "sot_grad_x": [P, P, P, P, i, i, i, i, P, P, f, P, P],
        "sot_cost_grad": [P, P, P, P, i, i, i, i, P, P, f, P, P, P],
        "sot_plan_coo": [P, P, P, P, i, i, i, i, P, P, f, f, i, ll, P, P, P, P, C.POINTER(ll), P],
        "sot_grad_x_coo": [P, P, i, i, i, i, P, P, P, P, P, P],
        "sot_check_inputs": [P, P, P, P, i, i, i, i, P],
        "sot_profile_enable": [i],
        "sot_profile_read": [C.POINTER(ll), C.POINTER(C.c_double)],
        "sot_profile_read_kinds": [C.POINTER(ll), C.POINTER(C.c_double)],
        "sot_status_string": [i],
        "sot_last_error": [],
        "sot_version": [],
        "sot_kernel_launches": [],
        "sot_select_path": [i, i],
        "sot_potentials_noalloc": [P, P, P, P, i, i, i, i, f, i, P, P, P],
        "sot_transport_apply": [P, P, P, P, i, i, i, i, P, P, f, P, i, i, P, i, P],
        "sot_grad_y": [P, P, P, P, i, i, i, i, P, P, f, P, i, P],
        "sot_apml_coo": [P, P, P, P, i, i, i, i, P, P, P, ll, f, i, P, P, P, P],
        "sot_async_status": [P],
        "sot_hvp": [P, P, P, P, i, i, i, i, P, P, f, P, i, f, P, i, P],
        "sot_test_hold_tile": [i, i, ll],
        "sot_plan_coo_operands": [P, P, P, P, i, i, i, i, P, P, f, f, P, P, P, P, P, P, P, P,
                                  C.POINTER(C.c_float), P],
    }
    for name, args in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = C.c_char_p if name in ("sot_status_string", "sot_last_error") else \
            (C.c_longlong if name == "sot_kernel_launches" else C.c_int)
    if path is None:
        _lib = L
    return L


def _check(rc: int, func: str):
    if rc != SOT_OK:
        L = load()
        raise SotError(rc, func, L.sot_last_error().decode() or L.sot_status_string(rc).decode())


def _ptr(t):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError("expected a torch.Tensor")
    if t.dtype != torch.float32 and t.dtype not in (torch.int32, torch.int64):
        raise TypeError(f"expected float32, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _want(t, name, count, dev, dtype=torch.float32):
    """A tensor the caller supplies must be contiguous, of ``dtype``, on ``dev``
    and hold exactly ``count`` elements (None: any count), since the library
    reads or writes that many."""
    if t is None:
        return t
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if count is not None and t.numel() != count:
        raise ValueError(f"{name} must hold {count} elements, got shape {tuple(t.shape)}")
    if t.device != dev:
        raise ValueError(f"{name} must be on {dev}, got {t.device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _shapes(X, Y, a, b):
    if not isinstance(X, torch.Tensor) or not isinstance(Y, torch.Tensor):
        raise TypeError("X and Y must be torch.Tensors")
    if X.dim() == 2:
        X = X.unsqueeze(0)
    if Y.dim() == 2:
        Y = Y.unsqueeze(0)
    if X.dim() != 3 or Y.dim() != 3:
        raise ValueError("X must be [B,n,d] or [n,d], Y [B,m,d] or [m,d]")
    B, n, d = X.shape
    B2, m, d2 = Y.shape
    if B != B2 or d != d2:
        raise ValueError("X [B,n,d] and Y [B,m,d] disagree")
    if a is not None and tuple(a.shape) not in ((B, n), (n,) if B == 1 else (B, n)):
        raise ValueError("a must be [B, n]")
    if b is not None and tuple(b.shape) not in ((B, m), (m,) if B == 1 else (B, m)):
        raise ValueError("b must be [B, m]")
    dev = X.device
    _want(X, "X", B * n * d, dev)
    _want(Y, "Y", B * m * d, dev)
    _want(a, "a", B * n, dev)
    _want(b, "b", B * m, dev)
    return X, Y, B, n, m, d


def _potentials_args(f, g, B, n, m, dev):
    return _want(f, "f", B * n, dev), _want(g, "g", B * m, dev)


def sot_version() -> int:
    return int(load().sot_version())


def sot_kernel_launches() -> int:
    return int(load().sot_kernel_launches())


def sot_select_path(d: int, flags: int = 0) -> int:
    """0 = fp32 point kernels, 1 = fp32 dense kernels, 2 = tensor-core kernels (negative: none)."""
    return int(load().sot_select_path(int(d), int(flags)))


def sot_status_string(status: int) -> str:
    return load().sot_status_string(int(status)).decode()


def sot_potentials(X, Y, a=None, b=None, eps=0.1, iters=100, f=None, g=None, stream=None):
    """Fixed schedule from f = g = 0; returns (f [B,n], g [B,m])."""
    X, Y, B, n, m, d = _shapes(X, Y, a, b)
    f = torch.empty(B, n, device=X.device, dtype=torch.float32) if f is None else f
    g = torch.empty(B, m, device=X.device, dtype=torch.float32) if g is None else g
    _potentials_args(f, g, B, n, m, X.device)
    rc = load().sot_potentials(_ptr(X), _ptr(Y), _ptr(a), _ptr(b), B, n, m, d, float(eps), int(iters), _ptr(f),
                               _ptr(g), _stream(stream))
    _check(rc, "sot_potentials")
    return f, g


def sot_potentials_noalloc(X, Y, a=None, b=None, eps=0.1, iters=100, f=None, g=None, stream=None):
    """sot_potentials for d <= 3 using the library's static scratch (no device
    allocation inside the call; see include/sot.h).  Pass preallocated f, g to
    keep this call path free of allocations on the Python side too."""
    X, Y, B, n, m, d = _shapes(X, Y, a, b)
    f = torch.empty(B, n, device=X.device, dtype=torch.float32) if f is None else f
    g = torch.empty(B, m, device=X.device, dtype=torch.float32) if g is None else g
    _potentials_args(f, g, B, n, m, X.device)
    rc = load().sot_potentials_noalloc(_ptr(X), _ptr(Y), _ptr(a), _ptr(b), B, n, m, d, float(eps), int(iters),
                                       _ptr(f), _ptr(g), _stream(stream))
    _check(rc, "sot_potentials_noalloc")
    return f, g


def sot_potentials_ex(X, Y, a=None, b=None, eps=0.1, eps_init=None, eps_factor=0.5, iters_per_stage=100,
                      max_iters=0, tol=0.0, flags=0, f=None, g=None, stats=False, stream=None):
    """General schedule (see sot_schedule in sot.h).  With ``flags & SOT_WARM_START``
    the given f, g are the initial potentials.  Returns (f, g) or (f, g, stats dict)."""
    X, Y, B, n, m, d = _shapes(X, Y, a, b)
    if flags & SOT_WARM_START and (f is None or g is None):
        raise ValueError("warm start needs f and g")
    f = torch.empty(B, n, device=X.device, dtype=torch.float32) if f is None else f
    g = torch.empty(B, m, device=X.device, dtype=torch.float32) if g is None else g
    _potentials_args(f, g, B, n, m, X.device)
    s = sot_schedule(float(eps), float(eps if eps_init is None else eps_init), float(eps_factor),
                     int(iters_per_stage), int(max_iters), float(tol), int(flags))
    st = None
    if stats:
        cap = 100000
        err = (C.c_float * max(B, 1))()
        si = (C.c_int * cap)()
        st = sot_stats(0, 0, 0, 0.0, C.cast(err, C.POINTER(C.c_float)), C.cast(si, C.POINTER(C.c_int)), cap)
    rc = load().sot_potentials_ex(_ptr(X), _ptr(Y), _ptr(a), _ptr(b), B, n, m, d, C.byref(s), _ptr(f), _ptr(g),
                                  C.byref(st) if st is not None else None, _stream(stream))
    _check(rc, "sot_potentials_ex")
    if not stats:
        return f, g
    info = dict(iters_done=st.iters_done, stages_done=st.stages_done, converged=bool(st.converged),
                final_eps=st.final_eps, err=[err[k] for k in range(B)],
                stage_iters=[si[k] for k in range(st.stages_done)])
    return f, g, info


def sot_plan_apply(X, Y, a, b, f, g, eps, cost=True, grad=True, rowsum=False, flags=0, stream=None):
    """Returns (cost [B] or None, grad [B,n,d] or None, rowsum [B,n] or None).
    Each of cost, grad, rowsum is True (allocate), False/None (skip) or a
    preallocated tensor to write into."""
    X, Y, B, n, m, d = _shapes(X, Y, a, b)
    dev = X.device
    pick = lambda want, shape: torch.empty(*shape, device=dev, dtype=torch.float32) if want is True else \
        (None if want is None or want is False else want)
    c, gr, r = pick(cost, (B,)), pick(grad, (B, n, d)), pick(rowsum, (B, n))
    _potentials_args(f, g, B, n, m, dev)
    _want(c, "cost", B, dev)
    _want(gr, "grad", B * n * d, dev)
    _want(r, "rowsum", B * n, dev)
    rc = load().sot_plan_apply(_ptr(X), _ptr(Y), _ptr(a), _ptr(b), B, n, m, d, _ptr(f), _ptr(g), float(eps),
                               _ptr(c), _ptr(gr), _ptr(r), int(flags), _stream(stream))
    _check(rc, "sot_plan_apply")
    return c, gr, r


def sot_transport_apply(X, Y, a, b, f, g, eps, V, side=0, flags=0, out=None, stream=None):
    """Transport-matrix product: side 0 -> P V with V [B,m,c] (out [B,n,c]);
    side 1 -> P^T V with V [B,n,c] (out [B,m,c]).  A [B,rows] V is one column."""
    X, Y, B, n, m, d = _shapes(X, Y, a, b)
    vec = V.dim() == 2
    V3 = V.unsqueeze(-1) if vec else V
    if V3.dtype != torch.float32 or not V3.is_contiguous() or V3.device != X.device:
        raise ValueError("V must be a contiguous float32 tensor on the device of X")
    rows_in, rows_out = (m, n) if side == 0 else (n, m)
    if V3.shape[0] != B or V3.shape[1] != rows_in:
        raise ValueError(f"V must have shape [B, {rows_in}, c] for side {side}")
    c = V3.shape[2]
    o = torch.empty(B, rows_out, c, device=X.device, dtype=torch.float32) if out is None else out
    _potentials_args(f, g, B, n, m, X.device)
    _want(o, "out", B * rows_out * c, X.device)
    rc = load().sot_transport_apply(_ptr(X), _ptr(Y), _ptr(a), _ptr(b), B, n, m, d, _ptr(f), _ptr(g),
                                    float(eps), _ptr(V3), int(c), int(side), _ptr(o), int(flags), _stream(stream))
    _check(rc, "sot_transport_apply")
    return o[..., 0] if vec else o


def sot_grad_y(X, Y, a, b, f, g, eps, flags=0, out=None, stream=None):
    """Gradient with respect to Y: 2 (b_j y_j - sum_i P_ij x_i), [B, m, d]."""
    X, Y, B, n, m, d = _shapes(X, Y, a, b)
    o = torch.empty(B, m, d, device=X.device, dtype=torch.float32) if out is None else out
    _potentials_args(f, g, B, n, m, X.device)
    _want(o, "out", B * m * d, X.device)
    rc = load().sot_grad_y(_ptr(X), _ptr(Y), _ptr(a), _ptr(b), B, n, m, d, _ptr(f), _ptr(g), float(eps), _ptr(o),
                           int(flags), _stream(stream))
    _check(rc, "sot_grad_y")
    return o


def sot_hvp(X, Y, a, b, f, g, eps, V, cg_iters=300, cg_tol=1e-5, out=None, stream=None):
    """Hessian-vector product of the entropic OT loss with respect to X at the
    potentials (f, g), applied to V [B, n, d]; returns H V [B, n, d]."""
    X, Y, B, n, m, d = _shapes(X, Y, a, b)
    _potentials_args(f, g, B, n, m, X.device)
    _want(V, "V", B * n * d, X.device)
    o = torch.empty(B, n, d, device=X.device, dtype=torch.float32) if out is None else out
    _want(o, "out", B * n * d, X.device)
    rc = load().sot_hvp(_ptr(X), _ptr(Y), _ptr(a), _ptr(b), B, n, m, d, _ptr(f), _ptr(g), float(eps), _ptr(V),
                        int(cg_iters), float(cg_tol), _ptr(o), 0, _stream(stream))
    _check(rc, "sot_hvp")
    return o


def sot_apml_coo(X, Y, a, b, coo, T, iters=10, loss=True, grad=True, stream=None):
    """Sparse APML on a stored support (``coo`` as sot_plan_coo returns it):
    returns (vals [nnz], loss [B] or None, grad [B,n,d] or None)."""
    X, Y, B, n, m, d = _shapes(X, Y, a, b)
    nnz = int(coo["nnz"])
    _want(coo["rows"], "coo rows", nnz, X.device, torch.int32)
    _want(coo["cols"], "coo cols", nnz, X.device, torch.int32)
    _want(coo["batch_offsets"], "coo batch_offsets", B + 1, X.device, torch.int64)
    vals = torch.empty(max(nnz, 1), device=X.device, dtype=torch.float32)
    lo = torch.empty(B, device=X.device, dtype=torch.float32) if loss else None
    gr = torch.empty(B, n, d, device=X.device, dtype=torch.float32) if grad else None
    rc = load().sot_apml_coo(_ptr(X), _ptr(Y), _ptr(a), _ptr(b), B, n, m, d, _ptr(coo["rows"]), _ptr(coo["cols"]),
                             _ptr(coo["batch_offsets"]), nnz, float(T), int(iters), _ptr(vals), _ptr(lo), _ptr(gr),
                             _stream(stream))
    _check(rc, "sot_apml_coo")
    return vals[:nnz], lo, gr


def sot_cost(X, Y, a, b, f, g, eps, stream=None):
    return sot_plan_apply(X, Y, a, b, f, g, eps, cost=True, grad=False, stream=stream)[0]


def sot_grad_x(X, Y, a, b, f, g, eps, stream=None):
    return sot_plan_apply(X, Y, a, b, f, g, eps, cost=False, grad=True, stream=stream)[1]


def sot_cost_grad(X, Y, a, b, f, g, eps, stream=None):
    c, gr, _ = sot_plan_apply(X, Y, a, b, f, g, eps, cost=True, grad=True, stream=stream)
    return c, gr


def sot_plan_coo(X, Y, a, b, f, g, eps, threshold=1e-8, dirs=3, capacity=None, stream=None):
    """Thresholded COO plan; returns dict(rows, cols, vals, batch_offsets, nnz).
    With capacity None the call runs twice if needed (count, then write)."""
    X, Y, B, n, m, d = _shapes(X, Y, a, b)
    dev = X.device
    _potentials_args(f, g, B, n, m, dev)
    L = load()
    off = torch.empty(B + 1, device=dev, dtype=torch.int64)
    nnz = C.c_longlong(0)
    cap = int(capacity) if capacity is not None else 0
    rows = torch.empty(max(cap, 1), device=dev, dtype=torch.int32)
    cols = torch.empty(max(cap, 1), device=dev, dtype=torch.int32)
    vals = torch.empty(max(cap, 1), device=dev, dtype=torch.float32)
    args = lambda: (_ptr(X), _ptr(Y), _ptr(a), _ptr(b), B, n, m, d, _ptr(f), _ptr(g), float(eps), float(threshold),
                    int(dirs), cap, _ptr(rows), _ptr(cols), _ptr(vals), _ptr(off), C.byref(nnz), _stream(stream))
    rc = L.sot_plan_coo(*args())
    if rc == SOT_ERR_CAPACITY and capacity is None:
        cap = int(nnz.value)
        rows = torch.empty(max(cap, 1), device=dev, dtype=torch.int32)
        cols = torch.empty(max(cap, 1), device=dev, dtype=torch.int32)
        vals = torch.empty(max(cap, 1), device=dev, dtype=torch.float32)
        rc = L.sot_plan_coo(*args())
    if rc == SOT_ERR_CAPACITY:
        raise SotError(rc, "sot_plan_coo", f"capacity {cap} < nnz {nnz.value}")
    _check(rc, "sot_plan_coo")
    k = int(nnz.value)
    return dict(rows=rows[:k], cols=cols[:k], vals=vals[:k], batch_offsets=off, nnz=k)


def sot_plan_coo_operands(X, Y, a, b, f, g, eps, threshold=1e-8, stream=None):
    """The fp32 operands sot_plan_coo decides its support from; returns
    dict(xc, lwx, Lx, yc, lwy, Ly, Mr, Mc, kappa, log2tau)."""
    X, Y, B, n, m, d = _shapes(X, Y, a, b)
    dev = X.device
    _potentials_args(f, g, B, n, m, dev)
    L = load()
    out = dict(xc=torch.empty(B, n, d, device=dev), lwx=torch.empty(B, n, device=dev),
               Lx=torch.empty(B, n, device=dev), yc=torch.empty(B, m, d, device=dev),
               lwy=torch.empty(B, m, device=dev), Ly=torch.empty(B, m, device=dev),
               Mr=torch.empty(B, n, device=dev), Mc=torch.empty(B, m, device=dev))
    sc = (C.c_float * 2)()
    rc = L.sot_plan_coo_operands(_ptr(X), _ptr(Y), _ptr(a), _ptr(b), B, n, m, d, _ptr(f), _ptr(g), float(eps),
                                 float(threshold), *(_ptr(out[k]) for k in ("xc", "lwx", "Lx", "yc", "lwy", "Ly",
                                                                            "Mr", "Mc")),
                                 sc, _stream(stream))
    _check(rc, "sot_plan_coo_operands")
    out["kappa"], out["log2tau"] = float(sc[0]), float(sc[1])
    return out


def sot_grad_x_coo(X, Y, rows, cols, vals, batch_offsets, grad=None, stream=None):
    X, Y, B, n, m, d = _shapes(X, Y, None, None)
    dev = X.device
    _want(rows, "rows", None, dev, torch.int32)
    _want(cols, "cols", rows.numel(), dev, torch.int32)
    _want(vals, "vals", rows.numel(), dev)
    _want(batch_offsets, "batch_offsets", B + 1, dev, torch.int64)
    grad = torch.empty(B, n, d, device=X.device, dtype=torch.float32) if grad is None else grad
    _want(grad, "grad", B * n * d, dev)
    rc = load().sot_grad_x_coo(_ptr(X), _ptr(Y), B, n, m, d, _ptr(rows), _ptr(cols), _ptr(vals),
                               _ptr(batch_offsets), _ptr(grad), _stream(stream))
    _check(rc, "sot_grad_x_coo")
    return grad


def sot_async_status(stream=None):
    """Raises SotError(SOT_ERR_TIMEOUT) when a bounded device-side wait gave up
    in an asynchronous call since the last check on this device; clears it."""
    _check(load().sot_async_status(_stream(stream)), "sot_async_status")


def sot_test_hold_tile(tile: int, after_launches: int = 0, wait_ns: int = 0):
    """Testing hook: after `after_launches` more tensor-core launches, those
    kernels withhold column tile `tile` of their chunk onward (tile < 0: off),
    so their waits run out after wait_ns nanoseconds."""
    _check(load().sot_test_hold_tile(int(tile), int(after_launches), int(wait_ns)), "sot_test_hold_tile")


def sot_check_inputs(X, Y, a=None, b=None, stream=None) -> int:
    """Returns the status code (0 ok, SOT_ERR_NONFINITE, ...) without raising."""
    X, Y, B, n, m, d = _shapes(X, Y, a, b)
    return int(load().sot_check_inputs(_ptr(X), _ptr(Y), _ptr(a), _ptr(b), B, n, m, d, _stream(stream)))


def sot_profile_enable(on: bool = True):
    _check(load().sot_profile_enable(int(bool(on))), "sot_profile_enable")


def sot_profile_read():
    """(half-step launches, total milliseconds) since the last read."""
    n = C.c_longlong(0)
    ms = C.c_double(0)
    _check(load().sot_profile_read(C.byref(n), C.byref(ms)), "sot_profile_read")
    return int(n.value), float(ms.value)


def sot_profile_read_kinds():
    """{"full": (half-steps, ms), "screened": (...), "cluster": (...)} since the last read."""
    n = (C.c_longlong * 3)()
    ms = (C.c_double * 3)()
    _check(load().sot_profile_read_kinds(n, ms), "sot_profile_read_kinds")
    return {"full": (int(n[0]), float(ms[0])), "screened": (int(n[1]), float(ms[1])),
            "cluster": (int(n[2]), float(ms[2]))}
