"""CPU oracle for the MXFP4 / NVFP4 block-scaled GEMM and BF16 quantizer.

TEST INFRASTRUCTURE ONLY.  The product path (the CUDA library and its Python
binding) never imports, links or runs anything in this package.  Only the
tests, the smoke check in the entry module and the CPU-baseline leg of the
benchmark use it.

The arithmetic lives in ``mx_oracle.c`` (plain C99, binary64 accumulation,
built with ``-ffp-contract=off``); this module builds it with gcc and wraps it
with ctypes + numpy.  It shares no code with the CUDA library.  Every
function's definition and the page passage it follows are stated in the C
file's header comment and at each function.

Pinned by the ``-m "not gpu"`` tests (``tests/test_oracle_*.py``): exhaustive
E2M1/E4M3/BF16 codec checks against brute-force nearest-value searches and
library routines, the exhaustive BF16 quantize sweep, GEMM brute force against
a dequantize-then-fp64 matmul, the closed-form invariants, and for the
stochastic-rounding path the published Philox4x32 known answers, exact
rational rounding and the half-way inputs that expose the draw layout, and for
the GEMM epilogue the normal CDF at known points, scipy's normal CDF and the
reflection identity of GELU.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")

FMT_MXFP4 = 0
FMT_NVFP4 = 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile mx_oracle.c into oracle/_build/liboracle.so (gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-fopenmp",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c_u8p = ctypes.POINTER(ctypes.c_uint8)
        c_u16p = ctypes.POINTER(ctypes.c_uint16)
        c_u32p = ctypes.POINTER(ctypes.c_uint32)
        c_i64 = ctypes.c_int64
        c_i64p = ctypes.POINTER(ctypes.c_int64)
        c_f64p = ctypes.POINTER(ctypes.c_double)
        lib.oracle_e2m1_decode.restype = ctypes.c_double
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint32]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint32
        lib.oracle_e2m1_encode.argtypes = [ctypes.c_double]
        lib.oracle_bf16_to_float.restype = ctypes.c_float
        lib.oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_floor_log2.restype = ctypes.c_int
        lib.oracle_bf16_floor_log2.argtypes = [ctypes.c_uint16]
        lib.oracle_ue8m0_decode.restype = ctypes.c_double
        lib.oracle_ue8m0_decode.argtypes = [ctypes.c_uint32]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint32]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint32
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.oracle_round_bf16.restype = ctypes.c_uint16
        lib.oracle_round_bf16.argtypes = [ctypes.c_double]
        lib.oracle_round_bf16_array.restype = None
        lib.oracle_round_bf16_array.argtypes = [c_f64p, c_i64, c_u16p]
        lib.oracle_mx_quantize.restype = None
        lib.oracle_mx_quantize.argtypes = [c_u16p, c_i64, c_i64, c_i64, c_u8p, c_u8p]
        lib.oracle_bf16_amax.restype = ctypes.c_float
        lib.oracle_bf16_amax.argtypes = [c_u16p, c_i64, c_i64, c_i64]
        lib.oracle_nvfp4_quantize.restype = None
        lib.oracle_nvfp4_quantize.argtypes = [c_u16p, c_i64, c_i64, c_i64, c_u8p, c_u8p,
                                              ctypes.POINTER(ctypes.c_float)]
        lib.oracle_block_gemm.restype = None
        lib.oracle_philox4x32.argtypes = [c_u32p, c_u32p, ctypes.c_int, c_u32p]
        lib.oracle_philox4x32.restype = None
        lib.oracle_e2m1_encode_sr.argtypes = [ctypes.c_double, ctypes.c_uint32]
        lib.oracle_e2m1_encode_sr.restype = ctypes.c_uint32
        lib.oracle_nvfp4_quantize_sr.argtypes = [c_u16p, c_i64, c_i64, c_i64, ctypes.c_uint64,
                                                 ctypes.c_int, ctypes.c_uint32, c_u8p, c_u8p,
                                                 ctypes.POINTER(ctypes.c_float)]
        lib.oracle_nvfp4_quantize_sr.restype = None
        lib.oracle_gelu.argtypes = [ctypes.c_double]
        lib.oracle_gelu.restype = ctypes.c_double
        lib.oracle_gemm_epilogue.argtypes = [c_f64p, c_i64, c_i64, ctypes.POINTER(ctypes.c_float),
                                             ctypes.c_int, ctypes.c_double, c_f64p, c_f64p]
        lib.oracle_gemm_epilogue.restype = None
        lib.oracle_block_gemm.argtypes = [ctypes.c_int, c_u8p, c_u8p, c_u8p, c_u8p,
                                          c_i64, c_i64, c_i64, ctypes.c_float, ctypes.c_float,
                                          c_i64p, c_i64, c_i64p, c_i64, c_f64p, c_f64p]
        lib.oracle_scale_tile.restype = None
        lib.oracle_scale_tile.argtypes = [c_u8p, c_i64, c_i64, c_u8p]
        _lib = lib
        return lib


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


# ----------------------------------------------------------------- codecs

def e2m1_decode(code: int) -> float:
    return _load().oracle_e2m1_decode(int(code))


def e2m1_encode(y: float) -> int:
    return _load().oracle_e2m1_encode(float(y))


def bf16_to_float(bits: int) -> float:
    return _load().oracle_bf16_to_float(int(bits))


def bf16_floor_log2(bits: int) -> int:
    return _load().oracle_bf16_floor_log2(int(bits))


def ue8m0_decode(e: int) -> float:
    return _load().oracle_ue8m0_decode(int(e))


def e4m3_decode(b: int) -> float:
    return _load().oracle_e4m3_decode(int(b))


def e4m3_encode(v: float) -> int:
    return _load().oracle_e4m3_encode(float(v))


def round_bf16(d: np.ndarray) -> np.ndarray:
    """Round binary64 values to BF16 (ties to even), returned as uint16 bits."""
    flat = np.ascontiguousarray(d, dtype=np.float64).ravel()
    out = np.empty(flat.shape, dtype=np.uint16)
    _load().oracle_round_bf16_array(_ptr(flat, ctypes.c_double), flat.size,
                                    _ptr(out, ctypes.c_uint16))
    return out.reshape(np.shape(d))


# ----------------------------------------------------------------- quantizers

def mx_quantize(x_bits: np.ndarray):
    """BF16 bits [rows, cols] -> (codes [rows, cols/2] u8, scales [rows, cols/32] u8)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    assert cols % 32 == 0
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    scales = np.zeros((rows, cols // 32), dtype=np.uint8)
    _load().oracle_mx_quantize(_ptr(x, ctypes.c_uint16), rows, cols, cols,
                               _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8))
    return codes, scales


def mx_quantize_2d(x_bits: np.ndarray):
    """Bidimensional MXFP4 quantize of BF16 bits [rows, cols] (rows, cols % 32 == 0).

    Returns (codes, scales, codes_t, scales_t): the rowwise quantize of x
    (blocks of 32 along a row) and the rowwise quantize of x transposed
    (blocks of 32 down a column of x), the latter stored as [cols, rows/2]
    codes and [cols, rows/32] scales.  This is the definition of the
    "rowwise + columnwise" output of NVIDIA/TransformerEngine #3809
    (NVFP4QuantizeBidimensionalG2RKernel: the columnwise result is the
    transposed output, passed as (cols, rows)), applied to the MX rule.
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    assert x.shape[0] % 32 == 0 and x.shape[1] % 32 == 0
    codes, scales = mx_quantize(x)
    codes_t, scales_t = mx_quantize(np.ascontiguousarray(x.T))
    return codes, scales, codes_t, scales_t


def bf16_amax(x_bits: np.ndarray) -> float:
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    return _load().oracle_bf16_amax(_ptr(x, ctypes.c_uint16), rows, cols, cols)


def nvfp4_quantize(x_bits: np.ndarray):
    """BF16 bits [rows, cols] -> (codes [rows, cols/2], E4M3 scales [rows, cols/16], s_t)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    assert cols % 16 == 0
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    scales = np.zeros((rows, cols // 16), dtype=np.uint8)
    s_t = ctypes.c_float(0.0)
    _load().oracle_nvfp4_quantize(_ptr(x, ctypes.c_uint16), rows, cols, cols,
                                  _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                                  ctypes.byref(s_t))
    return codes, scales, np.float32(s_t.value)


def philox4x32(ctr, key, rounds: int = 10) -> np.ndarray:
    """Philox4x32-``rounds`` of one 128-bit counter (4 x u32) under a 64-bit key (2 x u32)."""
    c = np.ascontiguousarray(ctr, dtype=np.uint32).reshape(4)
    k = np.ascontiguousarray(key, dtype=np.uint32).reshape(2)
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32(_ptr(c, ctypes.c_uint32), _ptr(k, ctypes.c_uint32), int(rounds),
                              _ptr(out, ctypes.c_uint32))
    return out


def e2m1_encode_sr(y: float, u: int) -> int:
    """Stochastic rounding of y to an E2M1 code with the uniform byte u."""
    return int(_load().oracle_e2m1_encode_sr(float(y), int(u)))


def nvfp4_quantize_sr(x_bits: np.ndarray, seed: int, rounds: int = 10, direction: int = 0):
    """NVFP4 quantize of BF16 bits [rows, cols] with stochastically rounded codes.

    Same s_t and scales as :func:`nvfp4_quantize`; block (r, j) draws
    Philox4x32-``rounds`` of counter (j, r, direction, 0) under the key
    (seed low, seed high) and element i of the block uses byte i of the draw.
    Returns (codes, scales, s_t).
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    assert cols % 16 == 0
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    scales = np.zeros((rows, cols // 16), dtype=np.uint8)
    s_t = ctypes.c_float(0.0)
    _load().oracle_nvfp4_quantize_sr(_ptr(x, ctypes.c_uint16), rows, cols, cols,
                                     int(seed) & 0xFFFFFFFFFFFFFFFF, int(rounds), int(direction),
                                     _ptr(codes, ctypes.c_uint8), _ptr(scales, ctypes.c_uint8),
                                     ctypes.byref(s_t))
    return codes, scales, np.float32(s_t.value)


def nvfp4_quantize_2d(x_bits: np.ndarray, seed=None, rounds: int = 10):
    """Bidimensional NVFP4 quantize of BF16 bits [rows, cols] (rows, cols % 16 == 0).

    Returns (codes, scales, codes_t, scales_t, s_t): the rowwise NVFP4
    quantize of x and that of x transposed (blocks of 16 down a column of x,
    stored as [cols, rows/2] codes and [cols, rows/16] scales), under the one
    tensor scale s_t = amax(x) / 2688 (x and x^T have the same amax).  The
    columnwise result is the transposed output of NVIDIA/TransformerEngine
    #3809 (NVFP4QuantizeBidimensionalG2RKernel, passed as (cols, rows)).
    With a seed the codes are rounded stochastically: the rowwise blocks draw
    with direction 0 and the columnwise blocks with direction 1 (the pages:
    one draw per output block, keyed by its coordinates and direction).
    """
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    assert x.shape[0] % 16 == 0 and x.shape[1] % 16 == 0
    xt = np.ascontiguousarray(x.T)
    if seed is None:
        codes, scales, s_t = nvfp4_quantize(x)
        codes_t, scales_t, s_tt = nvfp4_quantize(xt)
    else:
        codes, scales, s_t = nvfp4_quantize_sr(x, seed, rounds, direction=0)
        codes_t, scales_t, s_tt = nvfp4_quantize_sr(xt, seed, rounds, direction=1)
    assert s_t == s_tt
    return codes, scales, codes_t, scales_t, s_t


# ----------------------------------------------------------------- GEMM

def block_gemm(fmt: int, a_codes, a_scales, b_codes, b_scales, m: int, n: int, k: int,
               a_tensor_scale: float = 1.0, b_tensor_scale: float = 1.0,
               rows=None, cols=None):
    """D = A * B^T in binary64 for block-scaled FP4 operands (TN).

    Returns (d, s_abs), both [len(rows), len(cols)] float64, where s_abs is
    sum_k |a||b| (the scale of the rounding-error bounds).
    """
    lib = _load()
    a_codes = np.ascontiguousarray(a_codes, dtype=np.uint8)
    b_codes = np.ascontiguousarray(b_codes, dtype=np.uint8)
    a_scales = np.ascontiguousarray(a_scales, dtype=np.uint8)
    b_scales = np.ascontiguousarray(b_scales, dtype=np.uint8)
    blk = 32 if fmt == FMT_MXFP4 else 16
    assert a_codes.size == m * k // 2 and b_codes.size == n * k // 2
    assert a_scales.size == m * k // blk and b_scales.size == n * k // blk
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = m if r is None else r.size
    nc = n if c is None else c.size
    d = np.zeros((nr, nc), dtype=np.float64)
    s_abs = np.zeros((nr, nc), dtype=np.float64)
    lib.oracle_block_gemm(fmt, _ptr(a_codes, ctypes.c_uint8), _ptr(a_scales, ctypes.c_uint8),
                          _ptr(b_codes, ctypes.c_uint8), _ptr(b_scales, ctypes.c_uint8),
                          m, n, k, float(a_tensor_scale), float(b_tensor_scale),
                          None if r is None else _ptr(r, ctypes.c_int64), nr,
                          None if c is None else _ptr(c, ctypes.c_int64), nc,
                          _ptr(d, ctypes.c_double), _ptr(s_abs, ctypes.c_double))
    return d, s_abs


def mx_gemm(a_codes, a_scales, b_codes, b_scales, m, n, k, rows=None, cols=None):
    return block_gemm(FMT_MXFP4, a_codes, a_scales, b_codes, b_scales, m, n, k,
                      rows=rows, cols=cols)


def nvfp4_gemm(a_codes, a_scales, b_codes, b_scales, m, n, k, a_tensor_scale,
               b_tensor_scale, rows=None, cols=None):
    return block_gemm(FMT_NVFP4, a_codes, a_scales, b_codes, b_scales, m, n, k,
                      a_tensor_scale, b_tensor_scale, rows=rows, cols=cols)


# ----------------------------------------------------------------- scale order

def gelu(y: float) -> float:
    """GELU(y) = y * Phi(y) (erf form), binary64."""
    return float(_load().oracle_gelu(float(y)))


def gemm_epilogue(d, bias=None, gelu_on: bool = False, beta: float = 0.0, c=None) -> np.ndarray:
    """act(d + beta * c + bias[None, :]) in binary64 (act = GELU or identity).

    d: the GEMM result alpha * A * B^T, [m, n] (binary64); bias: FP32 [n] or
    None; c: the prior contents of D as values, [m, n], or None (no beta term).
    """
    d = np.ascontiguousarray(d, dtype=np.float64)
    m, n = d.shape
    out = np.empty_like(d)
    b = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    cc = None if c is None else np.ascontiguousarray(c, dtype=np.float64)
    _load().oracle_gemm_epilogue(_ptr(d, ctypes.c_double), m, n,
                                 None if b is None else _ptr(b, ctypes.c_float), int(bool(gelu_on)),
                                 float(beta), None if cc is None else _ptr(cc, ctypes.c_double),
                                 _ptr(out, ctypes.c_double))
    return out


def scale_tile(plain: np.ndarray) -> np.ndarray:
    """Plain scales [rows, kb] -> the 128x4 tiled order (flat uint8 array)."""
    p = np.ascontiguousarray(plain, dtype=np.uint8)
    rows, kb = p.shape
    rows_pad = (rows + 127) // 128 * 128
    kb_pad = (kb + 3) // 4 * 4
    out = np.zeros(rows_pad * kb_pad, dtype=np.uint8)
    _load().oracle_scale_tile(_ptr(p, ctypes.c_uint8), rows, kb, _ptr(out, ctypes.c_uint8))
    return out


def fp4_transpose(codes: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """Codes [rows, cols / 2] -> [cols, rows / 2] (the element-wise transpose of
    the FP4 matrix), both packed with element 2t of a row in the low nibble of
    byte t (R2).  "Integrate MXFP4 hipblaslt GEMM support", Takeaways: the
    operand layouts other than TN come down to the transpose of one operand;
    the scales, indexed by (operand row, K block), are not touched."""
    c = np.asarray(codes, dtype=np.uint8).reshape(rows, cols // 2)
    elems = np.empty((rows, cols), dtype=np.uint8)   # one code per entry
    elems[:, 0::2] = c & 0xF
    elems[:, 1::2] = c >> 4
    t = np.ascontiguousarray(elems.T)                # [cols, rows]
    return (t[:, 0::2] | (t[:, 1::2] << 4)).astype(np.uint8)


# ----------------------------------------------------------------- helpers

def e2m1_decode_array(codes: np.ndarray, k: int) -> np.ndarray:
    """Unpack codes [rows, k/2] to float64 element values [rows, k] (no scales).

    Element 2t is the low nibble of byte t, element 2t+1 the high nibble.
    """
    table = np.array([e2m1_decode(c) for c in range(16)], dtype=np.float64)
    c = np.asarray(codes, dtype=np.uint8)
    lo = table[c & 0xF]
    hi = table[c >> 4]
    out = np.empty(c.shape[:-1] + (k,), dtype=np.float64)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out
