"""GB300-native row normalisation: RMSNorm, LayerNorm and FusedAddRMSNorm,
forward and backward, as hand-written sm_103a CUDA kernels behind the C ABI
of include/gb300norm.h (libgb300norm.so), with a thin ctypes binding.

Import fails loudly if the library has not been built (there is no CPU path);
build it with ``row_normalization_rmsnorm_gb300.build.build()``.
"""
from ._binding import (  # noqa: F401
    CODE_DTYPE, DTYPE_CODE, LIB_PATH, NORM_BF16, NORM_F16, NORM_F32, NormError, SIGNATURES,
    lib, norm_bwd_workspace_bytes, norm_debug_launches, norm_debug_set_path, norm_debug_tune, norm_device_status, norm_fused_add_rms_bwd,
    norm_fused_add_rms_fwd, norm_ln_bwd, norm_ln_fwd, norm_rms_bwd, norm_rms_bwd_noalloc, norm_rms_fwd, norm_sum_ranks,
    status_str,
)
