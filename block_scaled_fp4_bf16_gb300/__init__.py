"""GB300 (sm_103a) MXFP4 / NVFP4 block-scaled GEMM and BF16 quantizer.

The compute path is the C-ABI library libmxfp4.so (include/mxfp4.h), built
from the CUDA sources in csrc/ by build.py; ``_binding`` exposes each entry
point under its C name.  Importing this package loads nothing: the library
is opened on the first call, and a call without it raises.
"""
from ._binding import (  # noqa: F401
    MX_ERR_ALIGNMENT, MX_ERR_CUDA, MX_ERR_DEVICE_TIMEOUT, MX_ERR_INVALID_ARG, MX_ERR_NOT_COMPILED,
    MX_ERR_UNSUPPORTED_ARCH, MX_ERR_UNSUPPORTED_FEATURE, MX_ERR_UNSUPPORTED_SHAPE,
    MX_ERR_WORKSPACE, MX_FMT_MXFP4, MX_FMT_NVFP4, MX_LAYOUT_TN, MX_OK, MX_OUT_BF16, MX_OUT_FP32,
    MX_SCALE_PLAIN, MX_SCALE_TCGEN05, MXError, lib, mx_available, mx_device_status,
    mx_error_string, mx_last_error_string, mx_gemm_workspace_bytes, mx_quantize_bf16,
    mx_quantize_workspace_bytes,
    mx_scale_bytes, mx_scale_relayout, mx_selftest_wait_timeout, mxfp4_gemm, nvfp4_gemm,
    mxfp4_gemm_static_workspace, MX_STATIC_WORKSPACE_BYTES, MX_QUANTIZE_GROUP_MAX,
    mx_quantize_tensor, mx_quantize_bf16_group, mx_quantize_group_workspace_bytes,
    mx_quantize_bf16_2d, nvfp4_quantize_bf16_sr, MX_PHILOX_MAX_ROUNDS, nvfp4_quantize_bf16_2d,
    mx_gemm_epilogue, mxfp4_gemm_ex, nvfp4_gemm_ex, mx_calibrate_mma, MX_MMA_MXF4,
    MX_MMA_MXF4NVF4_2X, MX_MMA_MXF4NVF4_4X, MX_CALIBRATE_MAX_STEPS, MX_ERR_DEVICE_BOUNDS,
    MX_BUILD_BOUNDS_CHECK, mx_build_flags, mx_fp4_transpose)
