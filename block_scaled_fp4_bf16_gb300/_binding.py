"""ctypes binding of the C ABI in include/mxfp4.h (argument marshalling only).

Every function here has the name of the C entry point it calls and does no
arithmetic of the method: pointers are taken from torch tensors (or plain
integer device addresses), the stream defaults to torch's current CUDA
stream, and a non-zero status raises MXError.  The shared library is loaded
on first use; if it is missing the call raises (there is no fallback path).
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
# The bounds-checked build (MX_BOUNDS_CHECK=1 in the environment) lives in its
# own folder, so the release library is never replaced by it.
LIB_PATH = os.path.join(_HERE, "_build_bounds" if os.environ.get("MX_BOUNDS_CHECK") == "1"
                        else "_build", "libmxfp4.so")

MX_OK = 0
MX_ERR_INVALID_ARG = -1
MX_ERR_NOT_COMPILED = -2
MX_ERR_UNSUPPORTED_ARCH = -3
MX_ERR_UNSUPPORTED_SHAPE = -4
MX_ERR_UNSUPPORTED_FEATURE = -5
MX_ERR_ALIGNMENT = -6
MX_ERR_WORKSPACE = -7
MX_ERR_CUDA = -8
MX_ERR_DEVICE_TIMEOUT = -9
MX_ERR_DEVICE_BOUNDS = -10

MX_FMT_MXFP4 = 0
MX_FMT_NVFP4 = 1
MX_SCALE_PLAIN = 0
MX_SCALE_TCGEN05 = 1
MX_LAYOUT_TN = 0
MX_OUT_BF16 = 0
MX_OUT_FP32 = 1
MX_STATIC_WORKSPACE_BYTES = 16 << 20
MX_QUANTIZE_GROUP_MAX = 8
MX_PHILOX_MAX_ROUNDS = 16
MX_MMA_MXF4 = 0
MX_MMA_MXF4NVF4_2X = 1
MX_MMA_MXF4NVF4_4X = 2
MX_CALIBRATE_MAX_STEPS = 1 << 20
MX_BUILD_BOUNDS_CHECK = 1

_lock = threading.Lock()
_lib = None


class mx_quantize_tensor(ctypes.Structure):
    """One tensor of mx_quantize_bf16_group (the C struct of the same name)."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ld_x", ctypes.c_int64), ("codes", ctypes.c_void_p),
                ("scales", ctypes.c_void_p), ("tensor_scale", ctypes.c_void_p)]


class mx_gemm_epilogue(ctypes.Structure):
    """include/mxfp4.h: optional GEMM epilogue (bias FP32 [n], beta * D_in, GELU)."""
    _fields_ = [("bias", ctypes.c_void_p), ("beta", ctypes.c_float), ("gelu", ctypes.c_int)]


class MXError(RuntimeError):
    def __init__(self, fn: str, code: int, detail: str = ""):
        self.code = code
        self.detail = detail
        super().__init__(f"{fn} failed: {code} ({mx_error_string(code)})"
                         + (f": {detail}" if detail else ""))


def lib() -> ctypes.CDLL:
    """Load libmxfp4.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        i64, vp, sz, i32 = ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int
        L.mx_error_string.restype = ctypes.c_char_p
        L.mx_error_string.argtypes = [i32]
        L.mx_last_error_string.restype = ctypes.c_char_p
        L.mx_last_error_string.argtypes = []
        L.mx_available.restype = i32
        L.mx_available.argtypes = []
        L.mx_build_flags.restype = i32
        L.mx_build_flags.argtypes = []
        L.mx_scale_bytes.restype = sz
        L.mx_scale_bytes.argtypes = [i64, i64, i32, i32]
        L.mx_quantize_workspace_bytes.restype = sz
        L.mx_quantize_workspace_bytes.argtypes = [i64, i64, i32]
        L.mx_quantize_bf16.restype = i32
        L.mx_quantize_bf16.argtypes = [vp, i64, i64, i64, i32, i32, vp, vp, vp, vp, sz, vp]
        L.mx_quantize_group_workspace_bytes.restype = sz
        L.mx_quantize_group_workspace_bytes.argtypes = [i32, i32]
        L.mx_quantize_bf16_group.restype = i32
        L.mx_quantize_bf16_group.argtypes = [ctypes.POINTER(mx_quantize_tensor), i32, i32, i32, vp,
                                             sz, vp]
        L.nvfp4_quantize_bf16_sr.restype = i32
        L.nvfp4_quantize_bf16_sr.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, ctypes.c_uint64,
                                             i32, vp, sz, vp]
        L.nvfp4_quantize_bf16_2d.restype = i32
        L.nvfp4_quantize_bf16_2d.argtypes = [vp, i64, i64, i64, i32, vp, vp, vp, vp, vp, i32,
                                             ctypes.c_uint64, i32, vp, sz, vp]
        L.mx_quantize_bf16_2d.restype = i32
        L.mx_quantize_bf16_2d.argtypes = [vp, i64, i64, i64, i32, i32, vp, vp, vp, vp, vp]
        ep = ctypes.POINTER(mx_gemm_epilogue)
        L.mxfp4_gemm_ex.restype = i32
        L.mxfp4_gemm_ex.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, i32, ep, vp, sz, vp]
        L.nvfp4_gemm_ex.restype = i32
        L.nvfp4_gemm_ex.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, i32, ep, vp,
                                    sz, vp]
        L.mx_scale_relayout.restype = i32
        L.mx_scale_relayout.argtypes = [vp, i64, i64, i32, vp, vp]
        L.mx_fp4_transpose.restype = i32
        L.mx_fp4_transpose.argtypes = [vp, i64, i64, vp, vp]
        L.mx_gemm_workspace_bytes.restype = sz
        L.mx_gemm_workspace_bytes.argtypes = [i64, i64, i64, i32]
        L.mxfp4_gemm.restype = i32
        L.mxfp4_gemm.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, i32, vp, sz, vp]
        L.nvfp4_gemm.restype = i32
        L.nvfp4_gemm.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, i32, vp, sz,
                                 vp]
        L.mxfp4_gemm_static_workspace.restype = i32
        L.mxfp4_gemm_static_workspace.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i32, i32,
                                                  i32, vp]
        L.mx_device_status.restype = i32
        L.mx_device_status.argtypes = [vp]
        L.mx_selftest_wait_timeout.restype = i32
        L.mx_selftest_wait_timeout.argtypes = [ctypes.c_uint64, vp]
        L.mx_calibrate_mma.restype = i32
        L.mx_calibrate_mma.argtypes = [i32, i32, i64, vp, i32, ctypes.POINTER(ctypes.c_double),
                                       ctypes.POINTER(i32), vp]
        _lib = L
        return L


def _ptr(x):
    """Device address of a tensor / int / None (NULL)."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _nbytes(x) -> int:
    if x is None:
        return 0
    return x.numel() * x.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, rc: int) -> int:
    if rc != MX_OK:
        raise MXError(fn, rc, mx_last_error_string())
    return rc


def mx_error_string(code: int) -> str:
    return lib().mx_error_string(code).decode()


def mx_last_error_string() -> str:
    """Detail of the last rejection or failure of a call on this thread."""
    return lib().mx_last_error_string().decode()


def mx_build_flags() -> int:
    """MX_BUILD_BOUNDS_CHECK when the loaded library is the bounds-checked build."""
    return int(lib().mx_build_flags())


def mx_available() -> bool:
    return bool(lib().mx_available())


def mx_scale_bytes(rows: int, cols: int, fmt: int, scale_layout: int) -> int:
    return lib().mx_scale_bytes(rows, cols, fmt, scale_layout)


def mx_quantize_workspace_bytes(rows: int, cols: int, fmt: int) -> int:
    return lib().mx_quantize_workspace_bytes(rows, cols, fmt)


def mx_gemm_workspace_bytes(m: int, n: int, k: int, split_k: int = 0) -> int:
    return lib().mx_gemm_workspace_bytes(m, n, k, split_k)


def mx_quantize_bf16(x, rows, cols, ld_x, fmt, scale_layout, codes, scales, tensor_scale=None,
                     workspace=None, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace) if not isinstance(workspace, int) else 0
    return _check("mx_quantize_bf16", lib().mx_quantize_bf16(
        _ptr(x), rows, cols, ld_x, fmt, scale_layout, _ptr(codes), _ptr(scales),
        _ptr(tensor_scale), _ptr(workspace), workspace_bytes, _stream(stream)))


def nvfp4_quantize_bf16_sr(x, rows, cols, ld_x, scale_layout, codes, scales, tensor_scale, seed,
                           philox_rounds=10, workspace=None, workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace) if not isinstance(workspace, int) else 0
    return _check("nvfp4_quantize_bf16_sr", lib().nvfp4_quantize_bf16_sr(
        _ptr(x), rows, cols, ld_x, scale_layout, _ptr(codes), _ptr(scales), _ptr(tensor_scale),
        int(seed) & 0xFFFFFFFFFFFFFFFF, philox_rounds, _ptr(workspace), workspace_bytes,
        _stream(stream)))


def mx_quantize_group_workspace_bytes(count: int, fmt: int) -> int:
    return lib().mx_quantize_group_workspace_bytes(count, fmt)


def mx_quantize_bf16_group(tensors, fmt, scale_layout, workspace=None, workspace_bytes=None,
                           stream=None):
    """tensors: sequence of (x, rows, cols, ld_x, codes, scales, tensor_scale) tuples."""
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace) if not isinstance(workspace, int) else 0
    arr = (mx_quantize_tensor * max(1, len(tensors)))()
    for i, (x, rows, cols, ld_x, codes, scales, tensor_scale) in enumerate(tensors):
        arr[i] = mx_quantize_tensor(_ptr(x), rows, cols, ld_x, _ptr(codes), _ptr(scales),
                                    _ptr(tensor_scale))
    return _check("mx_quantize_bf16_group", lib().mx_quantize_bf16_group(
        arr, len(tensors), fmt, scale_layout, _ptr(workspace), workspace_bytes, _stream(stream)))


def mx_quantize_bf16_2d(x, rows, cols, ld_x, fmt, scale_layout, codes, scales, codes_t, scales_t,
                        stream=None):
    return _check("mx_quantize_bf16_2d", lib().mx_quantize_bf16_2d(
        _ptr(x), rows, cols, ld_x, fmt, scale_layout, _ptr(codes), _ptr(scales), _ptr(codes_t),
        _ptr(scales_t), _stream(stream)))


def nvfp4_quantize_bf16_2d(x, rows, cols, ld_x, scale_layout, codes, scales, codes_t, scales_t,
                           tensor_scale, stochastic=0, seed=0, philox_rounds=10, workspace=None,
                           workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace) if not isinstance(workspace, int) else 0
    return _check("nvfp4_quantize_bf16_2d", lib().nvfp4_quantize_bf16_2d(
        _ptr(x), rows, cols, ld_x, scale_layout, _ptr(codes), _ptr(scales), _ptr(codes_t),
        _ptr(scales_t), _ptr(tensor_scale), int(stochastic), int(seed) & 0xFFFFFFFFFFFFFFFF,
        philox_rounds, _ptr(workspace), workspace_bytes, _stream(stream)))


def mx_scale_relayout(plain, rows, cols, fmt, tiled, stream=None):
    return _check("mx_scale_relayout", lib().mx_scale_relayout(
        _ptr(plain), rows, cols, fmt, _ptr(tiled), _stream(stream)))


def mx_fp4_transpose(codes, rows, cols, out, stream=None):
    return _check("mx_fp4_transpose", lib().mx_fp4_transpose(
        _ptr(codes), rows, cols, _ptr(out), _stream(stream)))


def mxfp4_gemm(a_codes, a_scales, b_codes, b_scales, d, m, n, k, layout=MX_LAYOUT_TN,
               out_dtype=MX_OUT_BF16, split_k=0, workspace=None, workspace_bytes=None,
               stream=None):
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace) if not isinstance(workspace, int) else 0
    return _check("mxfp4_gemm", lib().mxfp4_gemm(
        _ptr(a_codes), _ptr(a_scales), _ptr(b_codes), _ptr(b_scales), _ptr(d), m, n, k, layout,
        out_dtype, split_k, _ptr(workspace), workspace_bytes, _stream(stream)))


def nvfp4_gemm(a_codes, a_scales, b_codes, b_scales, a_tensor_scale, b_tensor_scale, d, m, n, k,
               layout=MX_LAYOUT_TN, out_dtype=MX_OUT_FP32, split_k=0, workspace=None,
               workspace_bytes=None, stream=None):
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace) if not isinstance(workspace, int) else 0
    return _check("nvfp4_gemm", lib().nvfp4_gemm(
        _ptr(a_codes), _ptr(a_scales), _ptr(b_codes), _ptr(b_scales), _ptr(a_tensor_scale),
        _ptr(b_tensor_scale), _ptr(d), m, n, k, layout, out_dtype, split_k, _ptr(workspace),
        workspace_bytes, _stream(stream)))


def _epilogue(bias, beta, gelu):
    if bias is None and not beta and not gelu:
        return None
    return ctypes.byref(mx_gemm_epilogue(_ptr(bias), float(beta), int(bool(gelu))))


def mxfp4_gemm_ex(a_codes, a_scales, b_codes, b_scales, d, m, n, k, layout=MX_LAYOUT_TN,
                  out_dtype=MX_OUT_BF16, split_k=0, bias=None, beta=0.0, gelu=False,
                  workspace=None, workspace_bytes=None, stream=None):
    """mxfp4_gemm with the epilogue D = act(A B^T + beta * D_in + bias)."""
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace) if not isinstance(workspace, int) else 0
    return _check("mxfp4_gemm_ex", lib().mxfp4_gemm_ex(
        _ptr(a_codes), _ptr(a_scales), _ptr(b_codes), _ptr(b_scales), _ptr(d), m, n, k, layout,
        out_dtype, split_k, _epilogue(bias, beta, gelu), _ptr(workspace), workspace_bytes,
        _stream(stream)))


def nvfp4_gemm_ex(a_codes, a_scales, b_codes, b_scales, a_tensor_scale, b_tensor_scale, d, m, n,
                  k, layout=MX_LAYOUT_TN, out_dtype=MX_OUT_FP32, split_k=0, bias=None, beta=0.0,
                  gelu=False, workspace=None, workspace_bytes=None, stream=None):
    """nvfp4_gemm with the epilogue D = act(alpha A B^T + beta * D_in + bias)."""
    if workspace_bytes is None:
        workspace_bytes = _nbytes(workspace) if not isinstance(workspace, int) else 0
    return _check("nvfp4_gemm_ex", lib().nvfp4_gemm_ex(
        _ptr(a_codes), _ptr(a_scales), _ptr(b_codes), _ptr(b_scales), _ptr(a_tensor_scale),
        _ptr(b_tensor_scale), _ptr(d), m, n, k, layout, out_dtype, split_k,
        _epilogue(bias, beta, gelu), _ptr(workspace), workspace_bytes, _stream(stream)))


def mxfp4_gemm_static_workspace(a_codes, a_scales, b_codes, b_scales, d, m, n, k,
                                layout=MX_LAYOUT_TN, out_dtype=MX_OUT_BF16, split_k=0,
                                stream=None):
    return _check("mxfp4_gemm_static_workspace", lib().mxfp4_gemm_static_workspace(
        _ptr(a_codes), _ptr(a_scales), _ptr(b_codes), _ptr(b_scales), _ptr(d), m, n, k, layout,
        out_dtype, split_k, _stream(stream)))


def mx_device_status(stream=None) -> int:
    """Synchronise the stream and return (not raise) the device status code."""
    return lib().mx_device_status(_stream(stream))


def mx_selftest_wait_timeout(timeout_ns: int, stream=None):
    return _check("mx_selftest_wait_timeout",
                  lib().mx_selftest_wait_timeout(timeout_ns, _stream(stream)))


def mx_calibrate_mma(form: int, pair: int, steps: int, cycles=None, stream=None):
    """Launch one calibration wave of block-scaled MMAs; returns (flops, units).
    cycles: None or a device tensor of >= SM-count int64 entries."""
    flops = ctypes.c_double(0.0)
    units = ctypes.c_int(0)
    cap = cycles.numel() if cycles is not None else 0
    _check("mx_calibrate_mma", lib().mx_calibrate_mma(
        form, pair, steps, _ptr(cycles), cap, ctypes.byref(flops), ctypes.byref(units),
        _stream(stream)))
    return flops.value, units.value
