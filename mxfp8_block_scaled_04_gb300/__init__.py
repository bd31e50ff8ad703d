"""GB300-native (sm_103a) MXFP8 block-scaled quantize engine.

BF16 [M, N] -> FP8 (E4M3 / E5M2) with one E8M0 scale per 32-element block,
rowwise (1x32) and columnwise (32x1) in one pass, with optional fused dbias
and a device noop flag, plus a grouped (MoE, ragged row offsets) variant.
The compute runs in the CUDA library built from ``csrc/``; this package is its
ctypes binding.
"""
from .binding import (  # noqa: F401
    BLOCK, E4M3, E5M2, MAX_GROUPS, MXFP8Error, MXFP8Tensor, STATUS_NAMES,
    lib, mxfp8_device_fault_word, mxfp8_kernel_launch_count, mxfp8_quantize,
    mxfp8_quantize_grouped, mxfp8_quantize_grouped_workspace_bytes, mxfp8_quantize_host,
    mxfp8_quantize_host_staging_bytes, mxfp8_quantize_dbias_noalloc, quantize_host,
    mxfp8_quantize_workspace_bytes, mxfp8_status_string, quantize, quantize_grouped, grouped_scale_col_rows,
    mxfp8_quantize_grouped_dbias, mxfp8_quantize_grouped_dbias_workspace_bytes,
    mxfp8_quantize_dact, quantize_dact, mxfp8_quantize_gated, quantize_gated, mxfp8_quantize_dgated,
    quantize_dgated, mxfp8_quantize_gated_grouped, quantize_gated_grouped, mxfp8_quantize_grouped_activated,
    mxfp8_quantize_grouped_swizzled, mxfp8_grouped_swizzled_scale_bytes, mxfp8_selftest_bounded_wait, mxfp8_activation_values,
    mxfp8_quantize_grouped_host, mxfp8_quantize_grouped_host_staging_bytes, mxfp8_grouped_host_chunks,
    quantize_grouped_host, mxfp8_quantize_ex_host, mxfp8_quantize_ex_host_staging_bytes,
    mxfp8_quantize_dact_host, mxfp8_quantize_dact_host_staging_bytes, quantize_dact_host,
    mxfp8_quantize_gated_host, mxfp8_quantize_gated_host_staging_bytes, quantize_gated_host,
    mxfp8_quantize_dgated_host, mxfp8_quantize_dgated_host_staging_bytes, quantize_dgated_host,
    QuantizeConfig, SCALES_PLAIN, SCALES_SWIZZLED, make_config, mxfp8_quantize_ex, mxfp8_scale_bytes,
)
