"""GB300-native memory-bound row reductions: softmax, RMSNorm and cross-entropy
forward over row-major M x N matrices, as hand-written sm_103a CUDA kernels
behind the C ABI in include/qk.h (libqk.so).

Importing this package loads nothing; the CUDA library is loaded on the first
call and a missing library raises.
"""
from .binding import (  # noqa: F401
    QK_BF16,
    QK_ERR_INVALID_ARG,
    QK_ERR_LAUNCH,
    QK_ERR_MISALIGNED,
    QK_ERR_NO_DEVICE,
    QK_ERR_TIMEOUT,
    QK_ERR_UNSUPPORTED,
    QK_F32,
    QK_OK,
    QK_OP_RMSNORM,
    QK_OP_SOFTMAX,
    QK_OP_XENT,
    QK_OP_RMSNORM_BWD,
    QK_OP_SOFTMAX_BWD,
    QK_OP_XENT_BWD,
    QkError,
    load_library,
    qk_get_device_status,
    qk_get_plan,
    qk_max_row_elements,
    qk_rmsnorm_bwd,
    qk_rmsnorm_bwd_workspace_size,
    qk_rmsnorm_fwd,
    qk_set_plan_override,
    qk_softmax_bwd,
    qk_softmax_fwd,
    qk_status_string,
    qk_test_wait_timeout,
    qk_xent_bwd,
    qk_xent_fwd,
    rmsnorm_bwd,
    rmsnorm_fwd,
    softmax_bwd,
    softmax_fwd,
    xent_bwd,
    xent_fwd,
)
