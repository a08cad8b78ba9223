"""GB300-native MoonEP layer path: plan, prefetch, permute, grouped GEMM,
combine and reduce_grad as sm_103a CUDA kernels behind a C ABI
(include/moonep.h); ``_lib`` is the ctypes binding with the same names."""
from ._lib import (  # noqa: F401
    GEMM_SCRATCH_BYTES, MoonepError, PlanWorkspace, dims, library, moonep_combine, moonep_combine_backward,
    moonep_dispatch, moonep_dispatch_backward, moonep_grouped_gemm_dw, moonep_grouped_gemm_dx,
    moonep_dispatch_send_once,
    moonep_get_plan_layout, moonep_grouped_gemm, moonep_launch_count, moonep_plan,
    moonep_plan_noalloc, moonep_plan_views, moonep_plan_workspace_bytes, moonep_prefetch_weights,
    moonep_read_status,
    moonep_reduce_grad, moonep_selftest_bounded_wait, status_string,
)
