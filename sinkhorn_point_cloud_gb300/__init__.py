"""GB300 (sm_103a) log-domain Sinkhorn for point clouds with squared-Euclidean cost.

The computation lives in libsot (C ABI: include/sot.h, CUDA sources in csrc/);
``binding`` marshals torch tensors into it, ``build`` compiles it in-tree and
``datagen`` draws the seeded synthetic workloads.
"""
from .binding import (sot_apml_coo, SOT_ERR_CAPACITY, SOT_ERR_CUDA, SOT_ERR_INVALID_ARG, SOT_ERR_NOMEM, SOT_ERR_NONFINITE,
                      SOT_ERR_TIMEOUT, SOT_ERR_UNSUPPORTED, SOT_OK, SOT_PREC_AUTO, SOT_PREC_F16X3, SOT_PREC_FP32,
                      SOT_COST_COSINE, SOT_NO_CLUSTER, SOT_STAGE_EARLY_EXIT, SOT_TC_NO_SCREEN, SOT_WARM_START, SotError,
                      sot_async_status, sot_check_inputs, sot_cost, sot_test_hold_tile,
                      sot_cost_grad, sot_grad_x, sot_grad_x_coo, sot_grad_y, sot_hvp, sot_kernel_launches, sot_select_path, sot_plan_apply,
                      sot_plan_coo, sot_plan_coo_operands, sot_potentials, sot_potentials_ex, sot_potentials_noalloc, sot_profile_enable,
                      sot_profile_read, sot_profile_read_kinds, sot_status_string, sot_transport_apply, sot_version)

__all__ = [n for n in dir() if n.startswith(("sot_", "SOT_", "Sot"))]
