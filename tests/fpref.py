"""Independent decoders used by the oracle's pins.

These restate the number formats from their bit-field definitions (or take a
library routine) so that the oracle's own tables and loops can be checked
against something other than themselves.  No oracle code is imported here.
"""
import math
from fractions import Fraction

import numpy as np


def e2m1_value(code: int) -> float:
    """E2M1 from its fields: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0."""
    s = (code >> 3) & 1
    e = (code >> 1) & 3
    m = code & 1
    mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
    return -mag if s else mag


E2M1_VALUES = np.array([e2m1_value(c) for c in range(16)], dtype=np.float64)


def decode_fp4_matrix(codes: np.ndarray, k: int) -> np.ndarray:
    """Packed codes [rows, k/2] -> values [rows, k] (even element = low nibble)."""
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty(c.shape[:-1] + (k,), dtype=np.float64)
    out[..., 0::2] = E2M1_VALUES[c & 0xF]
    out[..., 1::2] = E2M1_VALUES[c >> 4]
    return out


def ue8m0_value(e: int) -> float:
    return math.ldexp(1.0, int(e) - 127)


def e4m3_value(byte: int) -> float:
    """E4M3FN from its fields: bias 7, subnormals at exponent 0 (fields formula)."""
    s = (byte >> 7) & 1
    e = (byte >> 3) & 0xF
    m = byte & 7
    mag = (m / 8) * 2.0 ** -6 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
    return -mag if s else mag


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def nearest_e2m1_code(y: float) -> int:
    """Brute force over the 15 distinct E2M1 values with exact rationals.

    Ties go to the code with mantissa bit 0; |y| > 6 saturates to +-6; the
    sign of y is kept when the magnitude rounds to zero.
    """
    neg = math.copysign(1.0, y) < 0
    a = Fraction(abs(y))
    if a >= 6:
        return 7 | (8 if neg else 0)
    best, best_d = None, None
    for c in range(8):
        d = abs(a - Fraction(e2m1_value(c)))
        if best is None or d < best_d or (d == best_d and c % 2 == 0):
            best, best_d = c, d
    return best | (8 if neg else 0)


def nearest_e2m1_codes_vec(y: np.ndarray) -> np.ndarray:
    """Vectorised nearest-E2M1 search for values with few significant bits.

    Exact for inputs whose distance to every grid point is representable in
    binary64 (true for BF16 values scaled by a power of two).
    """
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    grid = E2M1_VALUES[:8]
    d = np.abs(a[..., None] - grid)
    dmin = d.min(axis=-1, keepdims=True)
    cand = d == dmin
    # among tied candidates prefer the even code
    even_pref = np.where(cand & (np.arange(8) % 2 == 0), 1, 0)
    has_even = even_pref.any(axis=-1)
    first_even = np.argmax(even_pref, axis=-1)
    first_any = np.argmax(cand, axis=-1)
    code = np.where(has_even, first_even, first_any)
    code = np.where(a >= 6.0, 7, code)
    sign = np.signbit(y).astype(np.int64) * 8
    return (code + sign).astype(np.uint8)
