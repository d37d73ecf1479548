"""Row-wise safe softmax on one GB300 (sm_103a): hand-written CUDA kernels
behind the C ABI of include/softmax.h, with a ctypes binding.

    import online_softmax_dispatcher_gb300 as osd
    y = osd.softmax(x)            # x: contiguous CUDA fp32 / fp16 / bf16 tensor

The raw C entry points are re-exported under their C names
(``softmax_fwd``, ``softmax_fwd_variant``, ...).  Nothing here computes a
softmax on the host: without the built library the calls raise
``SoftmaxLibraryMissing``.
"""
from ._binding import (  # noqa: F401
    BF16, EXPORTS, F16, F32, LIB_PATH, OK, VARIANTS, DeviceInfo, LaunchPlan, SoftmaxError,
    SoftmaxLibraryMissing, dtype_code, lib, plan_for, softmax, softmax_abi_version,
    softmax_device_query, softmax_fwd, softmax_fwd_plan, softmax_fwd_variant,
    softmax_get_device_error, softmax_last_cuda_error, softmax_plan, softmax_query_variant,
    softmax_selftest_bounded_wait, softmax_backward, softmax_bwd, softmax_bwd_variant, softmax_fwd_ws,
    softmax_workspace_size, softmax_fwd_noalloc, softmax_fwd_masked, softmax_fwd_masked_variant,
    softmax_masked, softmax_, layernorm_fwd, rmsnorm_fwd, norm_fwd_variant, layer_norm, rms_norm,
    LAYERNORM, RMSNORM, ERR_INVALID_ARG, ERR_UNSUPPORTED_DTYPE, ERR_ALIAS, ERR_CUDA, ERR_UNSUPPORTED_SHAPE,
    ERR_DEVICE_TIMEOUT, softmax_bwd_plan, softmax_masked_plan, norm_plan,
    softmax_strerror, softmax_variant_name,
)
