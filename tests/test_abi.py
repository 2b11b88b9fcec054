"""The C ABI library without a GPU: it builds, loads, exports every function
include/sot.h declares, and its host-side argument checks answer before any
CUDA call is made."""
import ctypes as C

import pytest

from sinkhorn_point_cloud_gb300 import binding, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def test_exports_every_declared_function(lib):
    names = binding.declared_functions()
    assert len(names) >= 14
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, f"declared but not exported: {missing}"


def test_version_and_status_strings(lib):
    assert lib.sot_version() == 100
    for code in range(0, -8, -1):
        s = lib.sot_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.sot_status_string(-99).decode() == "unknown status"


NULL = None


def test_invalid_sizes_rejected_on_host(lib):
    p = C.c_void_p(16)  # never dereferenced: the size check fails first
    assert lib.sot_potentials(p, p, NULL, NULL, 1, 0, 5, 3, 0.1, 10, p, p, NULL) == binding.SOT_ERR_INVALID_ARG
    assert b"n, m, d" in lib.sot_last_error()
    assert lib.sot_potentials(p, p, NULL, NULL, 1, 5, 0, 3, 0.1, 10, p, p, NULL) == binding.SOT_ERR_INVALID_ARG
    assert lib.sot_potentials(p, p, NULL, NULL, 1, 5, 5, 0, 0.1, 10, p, p, NULL) == binding.SOT_ERR_INVALID_ARG
    assert lib.sot_potentials(p, p, NULL, NULL, -1, 5, 5, 3, 0.1, 10, p, p, NULL) == binding.SOT_ERR_INVALID_ARG
    assert lib.sot_potentials(p, p, NULL, NULL, 1, 5, 5, 3, 0.1, -1, p, p, NULL) == binding.SOT_ERR_INVALID_ARG
    assert lib.sot_potentials(NULL, p, NULL, NULL, 1, 5, 5, 3, 0.1, 10, p, p, NULL) == binding.SOT_ERR_INVALID_ARG


def test_invalid_eps_and_flags_rejected(lib):
    p = C.c_void_p(16)
    for eps in (0.0, -1.0, float("nan"), float("inf")):
        assert lib.sot_potentials(p, p, NULL, NULL, 1, 5, 5, 3, eps, 10, p, p, NULL) == binding.SOT_ERR_INVALID_ARG
    s = binding.sot_schedule(0.1, 0.1, 0.5, 10, 10, 0.0, 1 << 12)
    assert lib.sot_potentials_ex(p, p, NULL, NULL, 1, 5, 5, 3, C.byref(s), p, p, NULL, NULL) == binding.SOT_ERR_INVALID_ARG
    assert lib.sot_potentials_ex(p, p, NULL, NULL, 1, 5, 5, 3, NULL, p, p, NULL, NULL) == binding.SOT_ERR_INVALID_ARG
    assert lib.sot_plan_apply(p, p, NULL, NULL, 1, 5, 5, 3, p, p, 0.0, p, p, NULL, 0, NULL) == binding.SOT_ERR_INVALID_ARG


def test_unsupported_precision_rejected(lib):
    p = C.c_void_p(16)
    s = binding.sot_schedule(0.1, 0.1, 0.5, 10, 10, 0.0, binding.SOT_PREC_F16X3)
    # d = 3 has no tensor-core path
    assert lib.sot_potentials_ex(p, p, NULL, NULL, 1, 5, 5, 3, C.byref(s), p, p, NULL, NULL) == binding.SOT_ERR_UNSUPPORTED
    # d = 1025 has no path at all
    assert lib.sot_potentials_ex(p, p, NULL, NULL, 1, 5, 5, 1025, C.byref(s), p, p, NULL, NULL) == binding.SOT_ERR_UNSUPPORTED
    s = binding.sot_schedule(0.1, 0.1, 0.5, 10, 10, 0.0, 0)
    assert lib.sot_potentials_ex(p, p, NULL, NULL, 1, 5, 5, 1025, C.byref(s), p, p, NULL, NULL) == binding.SOT_ERR_UNSUPPORTED


def test_coo_argument_checks(lib):
    p = C.c_void_p(16)
    nnz = C.c_longlong(123)
    assert lib.sot_plan_coo(p, p, NULL, NULL, 1, 5, 5, 3, p, p, 0.1, 1.5, 3, 10, p, p, p, p, C.byref(nnz), NULL) \
        == binding.SOT_ERR_INVALID_ARG
    assert nnz.value == 0
    assert lib.sot_plan_coo(p, p, NULL, NULL, 1, 5, 5, 3, p, p, 0.1, 1e-8, 0, 10, p, p, p, p, C.byref(nnz), NULL) \
        == binding.SOT_ERR_INVALID_ARG
    assert lib.sot_plan_coo(p, p, NULL, NULL, 1, 5, 5, 3, p, p, 0.1, 1e-8, 3, -1, p, p, p, p, C.byref(nnz), NULL) \
        == binding.SOT_ERR_INVALID_ARG
    assert lib.sot_plan_coo(p, p, NULL, NULL, 1, 5, 5, 3, p, p, 0.1, 1e-8, 3, 10, p, p, p, p, NULL, NULL) \
        == binding.SOT_ERR_INVALID_ARG


def test_empty_batch_is_a_no_op(lib):
    assert lib.sot_potentials(NULL, NULL, NULL, NULL, 0, 5, 5, 3, 0.1, 10, NULL, NULL, NULL) == binding.SOT_OK
    nnz = C.c_longlong(7)
    assert lib.sot_plan_coo(NULL, NULL, NULL, NULL, 0, 5, 5, 3, NULL, NULL, 0.1, 1e-8, 3, 0, NULL, NULL, NULL, NULL,
                            C.byref(nnz), NULL) == binding.SOT_OK
    assert nnz.value == 0


def test_python_binding_refuses_cpu_tensors():
    import torch
    X = torch.zeros(1, 4, 3)
    with pytest.raises(ValueError):
        binding.sot_potentials(X, X, eps=0.1, iters=1)


def test_transport_arguments_rejected_on_host(lib):
    p = C.c_void_p(16)
    tr = lib.sot_transport_apply
    ok = (p, p, NULL, NULL, 1, 5, 6, 3, p, p, 0.1, p)
    assert tr(*ok, 0, 0, p, 0, NULL) == binding.SOT_ERR_INVALID_ARG      # c = 0
    assert b"c must satisfy" in lib.sot_last_error()
    assert tr(*ok, 65, 0, p, 0, NULL) == binding.SOT_ERR_INVALID_ARG     # c above 64
    assert tr(*ok, 4, 2, p, 0, NULL) == binding.SOT_ERR_INVALID_ARG      # side 2
    assert tr(*ok, 4, 0, p, 1 << 3, NULL) == binding.SOT_ERR_INVALID_ARG  # unknown flag
    assert tr(*ok, 4, 0, NULL, 0, NULL) == binding.SOT_ERR_INVALID_ARG   # out NULL
    assert tr(p, p, NULL, NULL, 1, 5, 6, 3, p, p, 0.0, p, 4, 0, p, 0, NULL) == binding.SOT_ERR_INVALID_ARG
    assert tr(p, p, NULL, NULL, 1, 5, 6, 300, p, p, 0.1, p, 4, 0, p, 0, NULL) == binding.SOT_ERR_UNSUPPORTED
    assert tr(p, p, NULL, NULL, 0, 5, 6, 3, NULL, NULL, 0.1, NULL, 4, 0, NULL, 0, NULL) == binding.SOT_OK  # B = 0


def test_grad_y_arguments_rejected_on_host(lib):
    p = C.c_void_p(16)
    assert lib.sot_grad_y(p, p, NULL, NULL, 1, 5, 6, 3, p, p, 0.1, NULL, 0, NULL) == binding.SOT_ERR_INVALID_ARG
    assert lib.sot_grad_y(p, p, NULL, NULL, 1, 5, 6, 3, p, p, 0.1, p, 1 << 3, NULL) == binding.SOT_ERR_INVALID_ARG
    assert lib.sot_grad_y(p, p, NULL, NULL, 1, 5, 6, 300, p, p, 0.1, p, 0, NULL) == binding.SOT_ERR_UNSUPPORTED


def test_apml_arguments_rejected_on_host(lib):
    p = C.c_void_p(16)
    ap = lib.sot_apml_coo
    assert ap(p, p, NULL, NULL, 1, 5, 6, 3, p, p, p, 10, 0.0, 3, p, p, p, NULL) == binding.SOT_ERR_INVALID_ARG
    assert b"T must be" in lib.sot_last_error()
    assert ap(p, p, NULL, NULL, 1, 5, 6, 3, p, p, p, 10, 0.1, -1, p, p, p, NULL) == binding.SOT_ERR_INVALID_ARG
    assert ap(p, p, NULL, NULL, 1, 5, 6, 3, p, p, p, -1, 0.1, 3, p, p, p, NULL) == binding.SOT_ERR_INVALID_ARG
    assert ap(p, p, NULL, NULL, 1, 5, 6, 3, p, p, NULL, 10, 0.1, 3, p, p, p, NULL) == binding.SOT_ERR_INVALID_ARG
    assert ap(p, p, NULL, NULL, 0, 5, 6, 3, NULL, NULL, NULL, 0, 0.1, 3, NULL, NULL, NULL, NULL) == binding.SOT_OK


def test_python_binding_checks_caller_tensors():
    """Every tensor a caller supplies is checked for dtype, element count,
    device and layout before the library is called (CPU tensors of the right
    layout get as far as the device check)."""
    import torch
    B, n, m, d = 2, 5, 4, 3
    X, Y = torch.zeros(B, n, d), torch.zeros(B, m, d)
    f, g = torch.zeros(B, n), torch.zeros(B, m)
    with pytest.raises(TypeError, match="X"):
        binding.sot_potentials(X.to(torch.int32), Y, eps=0.1, iters=1)
    with pytest.raises(ValueError, match="f must hold 10"):
        binding.sot_potentials(X, Y, eps=0.1, iters=1, f=torch.zeros(B, n + 1), g=g)
    with pytest.raises(ValueError, match="g must hold 8"):
        binding.sot_plan_apply(X, Y, None, None, f, torch.zeros(m), 0.1)
    with pytest.raises(ValueError, match="grad must hold 30"):
        binding.sot_plan_apply(X, Y, None, None, f, g, 0.1, grad=torch.zeros(B, n, d + 1))
    with pytest.raises(ValueError, match="out must hold 20"):
        binding.sot_transport_apply(X, Y, None, None, f, g, 0.1, torch.zeros(B, m, 2), side=0,
                                    out=torch.zeros(B, n + 3, 2))
    with pytest.raises(ValueError, match="out must hold 24"):
        binding.sot_grad_y(X, Y, None, None, f, g, 0.1, out=torch.zeros(B, n, d))
    with pytest.raises(ValueError, match="contiguous"):
        binding.sot_grad_y(X, Y, None, None, f, g, 0.1, out=torch.zeros(B, d, m).transpose(1, 2))
    coo = dict(rows=torch.zeros(7, dtype=torch.int64), cols=torch.zeros(7, dtype=torch.int32),
               batch_offsets=torch.zeros(B + 1, dtype=torch.int64), nnz=7)
    with pytest.raises(TypeError, match="coo rows"):
        binding.sot_apml_coo(X, Y, None, None, coo, 0.1)
    coo["rows"] = torch.zeros(7, dtype=torch.int32)
    coo["batch_offsets"] = torch.zeros(B, dtype=torch.int64)
    with pytest.raises(ValueError, match="batch_offsets must hold 3"):
        binding.sot_apml_coo(X, Y, None, None, coo, 0.1)
    with pytest.raises(ValueError, match="vals must hold 7"):
        binding.sot_grad_x_coo(X, Y, coo["rows"], coo["cols"], torch.zeros(6), torch.zeros(B + 1, dtype=torch.int64))
    # a correct layout passes every check and stops at the device check
    with pytest.raises(ValueError, match="CUDA device"):
        binding.sot_plan_apply(X, Y, None, None, f, g, 0.1)


def test_path_selection(lib):
    """The kernel family each dimension and precision flag takes (host logic,
    no GPU needed): d <= 3 the point kernels; under automatic precision the
    fp32 kernels for 4 <= d <= 16 and the tensor cores for 17 <= d <= 1024
    (zero-padded to 64, 128, 192, 256, 512 or 1024); the fp16 split takes any
    4 <= d <= 1024; fp32 any d up to 1024; nothing goes past d = 1024."""
    point, dense, tensor = 0, 1, 2
    for d in (1, 2, 3):
        assert lib.sot_select_path(d, binding.SOT_PREC_AUTO) == point
        assert lib.sot_select_path(d, binding.SOT_PREC_FP32) == point
        assert lib.sot_select_path(d, binding.SOT_PREC_F16X3) == binding.SOT_ERR_UNSUPPORTED
    for d in (4, 8, 13, 16):
        assert lib.sot_select_path(d, binding.SOT_PREC_AUTO) == dense, d
        assert lib.sot_select_path(d, binding.SOT_PREC_F16X3) == tensor, d
        assert lib.sot_select_path(d, binding.SOT_PREC_FP32) == dense, d
    for d in (17, 63, 64, 65, 100, 128, 192, 200, 255, 256, 257, 320, 512, 1000, 1024):
        assert lib.sot_select_path(d, binding.SOT_PREC_AUTO) == tensor, d
        assert lib.sot_select_path(d, binding.SOT_PREC_F16X3) == tensor, d
        assert lib.sot_select_path(d, binding.SOT_PREC_FP32) == dense, d
    for flags in (binding.SOT_PREC_AUTO, binding.SOT_PREC_F16X3, binding.SOT_PREC_FP32):
        assert lib.sot_select_path(1025, flags) == binding.SOT_ERR_UNSUPPORTED


def test_hvp_arguments_rejected_on_host(lib):
    p = C.c_void_p(16)
    args = lambda d, it, tol, flags: (p, p, NULL, NULL, 1, 5, 5, d, p, p, 0.1, p, it, tol, p, flags, NULL)
    assert lib.sot_hvp(*args(10, 50, 1e-5, 0)) == binding.SOT_ERR_UNSUPPORTED  # d <= 9
    assert lib.sot_hvp(*args(3, 0, 1e-5, 0)) == binding.SOT_ERR_INVALID_ARG  # cg_iters >= 1
    assert lib.sot_hvp(*args(3, 50, -1.0, 0)) == binding.SOT_ERR_INVALID_ARG  # cg_tol >= 0
    assert lib.sot_hvp(*args(3, 50, 1e-5, 1)) == binding.SOT_ERR_INVALID_ARG  # no flags
    assert lib.sot_hvp(p, p, NULL, NULL, 1, 5, 5, 3, p, p, 0.1, NULL, 50, 1e-5, p, 0, NULL) == \
        binding.SOT_ERR_INVALID_ARG  # V must not be NULL
    assert lib.sot_hvp(p, p, NULL, NULL, 0, 5, 5, 3, NULL, NULL, 0.1, NULL, 50, 1e-5, NULL, 0, NULL) == binding.SOT_OK
