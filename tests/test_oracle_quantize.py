"""Pins of the oracle's MXFP4 and NVFP4 quantizers (CPU only)."""
import math

import numpy as np
import pytest

from block_scaled_fp4_bf16_gb300 import synth
from tests import fpref


def _unpack(codes, k):
    c = np.asarray(codes, dtype=np.uint8)
    out = np.empty(c.shape[:-1] + (k,), dtype=np.uint8)
    out[..., 0::2] = c & 0xF
    out[..., 1::2] = c >> 4
    return out


def _mx_exponent(amax: float) -> int:
    """Shared exponent from Python's frexp: floor(log2 amax) - 2, clamped."""
    if amax == 0.0:
        return -127
    return max(-127, min(127, math.frexp(amax)[1] - 1 - 2))


def _brute_force_mx(x_bits):
    """Independent MXFP4 quantizer: frexp exponent + exact nearest-grid search."""
    x = fpref.bf16_bits_to_f64(x_bits)
    rows, cols = x.shape
    blocks = x.reshape(rows, cols // 32, 32)
    amax = np.abs(blocks).max(axis=-1)
    e = np.vectorize(_mx_exponent, otypes=[np.int64])(amax)
    y = np.ldexp(blocks, -e[..., None])
    codes = fpref.nearest_e2m1_codes_vec(y).reshape(rows, cols)
    return codes, (e + 127).astype(np.uint8)


def _finite_bf16():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return b[((b >> 7) & 0xFF) != 0xFF]


def test_mx_quantize_exhaustive_bf16_as_block_max(oracle):
    """Every finite BF16 value as the largest element of its block."""
    v = _finite_bf16()
    x = np.zeros((v.size, 32), dtype=np.uint16)
    x[:, 0] = v
    x[:, 17] = v & 0x7FFF  # same magnitude, positive, in the high nibble of a byte
    codes, scales = oracle.mx_quantize(x)
    ref_codes, ref_scales = _brute_force_mx(x)
    assert np.array_equal(scales[:, 0], ref_scales[:, 0])
    assert np.array_equal(_unpack(codes, 32), ref_codes)


@pytest.mark.parametrize("anchor_exp", [-133, -126, -100, -20, -1, 0, 1, 3, 60, 127])
def test_mx_quantize_exhaustive_bf16_under_anchor(oracle, anchor_exp):
    """Every finite BF16 value in a block whose amax is set by another element."""
    v = _finite_bf16()
    anchor = synth.f32_to_bf16_bits(np.array([np.ldexp(1.75, anchor_exp)], np.float32))[0]
    x = np.zeros((v.size, 32), dtype=np.uint16)
    x[:, 3] = v
    x[:, 30] = anchor
    codes, scales = oracle.mx_quantize(x)
    ref_codes, ref_scales = _brute_force_mx(x)
    assert np.array_equal(scales[:, 0], ref_scales[:, 0])
    assert np.array_equal(_unpack(codes, 32), ref_codes)


def test_mx_quantize_random_blocks_brute_force(oracle):
    x = synth.bf16_normal(64, 512, 1.0, seed=11)
    x[5, :32] = 0                       # an all-zero block
    x[6, 32:64] = 0x8000                # a block of -0
    codes, scales = oracle.mx_quantize(x)
    ref_codes, ref_scales = _brute_force_mx(x)
    assert np.array_equal(scales, ref_scales)
    assert np.array_equal(_unpack(codes, 512), ref_codes)
    assert scales[5, 0] == 0 and np.all(_unpack(codes, 512)[5, :32] == 0)
    assert np.all(_unpack(codes, 512)[6, 32:64] == 8)


def test_mx_block_max_lands_in_top_binade(oracle):
    """Invariant of the shared-exponent rule: the block max maps to 4 or 6."""
    x = synth.bf16_normal(256, 1024, 1.0, seed=12)
    codes, scales = oracle.mx_quantize(x)
    mags = _unpack(codes, 1024).reshape(256, 32, 32) & 7
    assert np.all(mags.max(axis=-1) >= 6)


def test_mx_quantize_dequantize_round_trip(oracle):
    """quantize(dequantize(q, s)) == (q, s) when each block's max code is 4 or 6."""
    rng = np.random.default_rng(13)
    rows, k = 128, 256
    codes = rng.integers(0, 256, size=(rows, k // 2), dtype=np.uint8)
    u = _unpack(codes, k).reshape(rows, k // 32, 32)
    # force a magnitude-6 or magnitude-4 element into every block
    u[..., 0] = (u[..., 0] & 8) | rng.choice([6, 7], size=u.shape[:-1])
    u = u.reshape(rows, k)
    codes = (u[:, 0::2] | (u[:, 1::2] << 4)).astype(np.uint8)
    scales = rng.integers(110, 145, size=(rows, k // 32), dtype=np.uint8)
    vals = fpref.E2M1_VALUES[u] * np.repeat(np.ldexp(1.0, scales.astype(np.int64) - 127), 32, axis=1)
    x = synth.f32_to_bf16_bits(vals.astype(np.float32))  # exact: <= 2 significant bits
    assert np.array_equal(fpref.bf16_bits_to_f64(x), vals)
    q, s = oracle.mx_quantize(x)
    assert np.array_equal(s, scales)
    assert np.array_equal(q, codes)


def test_mx_nibble_order(oracle):
    x = np.zeros((1, 32), dtype=np.uint16)
    x[0, 0] = synth.f32_to_bf16_bits(np.array([1.0], np.float32))[0]
    x[0, 1] = synth.f32_to_bf16_bits(np.array([-6.0], np.float32))[0]
    codes, scales = oracle.mx_quantize(x)
    # amax 6 -> exponent floor(log2 6) - 2 = 0 -> scale 127; 1.0 -> code 2 (low nibble),
    # -6.0 -> code 15 (high nibble)
    assert scales[0, 0] == 127
    assert codes[0, 0] == (15 << 4) | 2


# ----------------------------------------------------------------- bidimensional MXFP4

def test_mx_quantize_2d_columnwise_brute_force(oracle):
    """The columnwise half against the independent brute-force quantizer run on
    the columns (blocks of 32 down a column), stored transposed."""
    x = synth.bf16_normal(96, 160, 1.0, seed=21)
    x[32:64, 7] = 0                     # an all-zero column block
    x[0:32, 9] = 0x8000                 # a column block of -0
    codes, scales, codes_t, scales_t = oracle.mx_quantize_2d(x)
    rc, rs = _brute_force_mx(x)
    assert np.array_equal(_unpack(codes, 160), rc) and np.array_equal(scales, rs)
    cc, cs = _brute_force_mx(np.ascontiguousarray(x.T))
    assert codes_t.shape == (160, 48) and scales_t.shape == (160, 3)
    assert np.array_equal(_unpack(codes_t, 96), cc) and np.array_equal(scales_t, cs)
    assert scales_t[7, 1] == 0 and np.all(_unpack(codes_t, 96)[7, 32:64] == 0)
    assert np.all(_unpack(codes_t, 96)[9, 0:32] == 8)


def test_mx_quantize_2d_orientation(oracle):
    """One non-zero element at (r, c): the rowwise code sits at row r, column c;
    the columnwise code at row c, column r of the transposed output."""
    r, c = 45, 70
    x = np.zeros((64, 96), dtype=np.uint16)
    x[r, c] = synth.f32_to_bf16_bits(np.array([-3.0], np.float32))[0]
    codes, scales, codes_t, scales_t = oracle.mx_quantize_2d(x)
    u, ut = _unpack(codes, 96), _unpack(codes_t, 64)
    # amax 3 -> exponent floor(log2 3) - 2 = -1 -> scale 126; -3 * 2 = -6 -> code 15
    assert u[r, c] == 15 and np.count_nonzero(u) == 1
    assert ut[c, r] == 15 and np.count_nonzero(ut) == 1
    assert scales[r, c // 32] == 126 and scales_t[c, r // 32] == 126
    assert np.count_nonzero(scales) == 1 and np.count_nonzero(scales_t) == 1


def test_mx_quantize_2d_symmetric_input(oracle):
    """For a symmetric matrix the two directions give the same bytes."""
    x = synth.bf16_normal(128, 128, 2.0, seed=22)
    x = np.triu(x) + np.triu(x, 1).T
    codes, scales, codes_t, scales_t = oracle.mx_quantize_2d(x)
    assert np.array_equal(codes, codes_t) and np.array_equal(scales, scales_t)


# ----------------------------------------------------------------- NVFP4

def test_nvfp4_exact_regime_reduces_to_nearest_grid(oracle):
    """With s_t and every block scale powers of two, no binary32 operation rounds,
    and the codes must be the nearest E2M1 values of x / (sb * s_t)."""
    rng = np.random.default_rng(21)
    rows, cols = 64, 256
    p = -3                               # s_t = 2^p exactly
    amax_t = 2688.0 * 2.0 ** p
    q = rng.integers(-6, 3, size=(rows, cols // 16))   # block amax = 6 * s_t * 2^q
    blk_amax = 6.0 * 2.0 ** p * np.ldexp(1.0, q)
    x = rng.uniform(-1, 1, size=(rows, cols // 16, 16)) * blk_amax[..., None]
    x[..., 0] = blk_amax                 # the block max, exactly
    x = x.reshape(rows, cols)
    x[0, :16] = 0
    x[0, 0] = amax_t                     # the tensor max, alone in its block
    xb = synth.f32_to_bf16_bits(x.astype(np.float32))
    xv = fpref.bf16_bits_to_f64(xb)
    assert xv[0, 0] == amax_t
    codes, scales, s_t = oracle.nvfp4_quantize(xb)
    assert s_t == np.float32(2.0 ** p)
    blocks = xv.reshape(rows, cols // 16, 16)
    ba = np.abs(blocks).max(axis=-1)
    # expected block scale: amax_b / (6 s_t) is a power of two for every block
    ratio = ba / (6.0 * 2.0 ** p)
    assert ratio[0, 0] == 448.0          # E4M3 max: y = 6 and zeros in that block
    lr = np.log2(ratio)
    lr[0, 0] = 0
    assert np.all(lr == np.round(lr))
    exp_scales = np.array([[oracle.e4m3_encode(r) for r in row] for row in ratio], np.uint8)
    for r in range(rows):
        for j in range(cols // 16):
            assert fpref.e4m3_value(int(scales[r, j])) == ratio[r, j]
    assert np.array_equal(scales, exp_scales)
    den = np.vectorize(fpref.e4m3_value)(scales.astype(np.int64)) * 2.0 ** p
    y = blocks / den[..., None]
    assert np.array_equal(_unpack(codes, cols), fpref.nearest_e2m1_codes_vec(y).reshape(rows, cols))


def test_nvfp4_random_properties(oracle):
    x = synth.bf16_normal(128, 1024, 1.0, seed=22)
    codes, scales, s_t = oracle.nvfp4_quantize(x)
    xv = fpref.bf16_bits_to_f64(x)
    amax_t = np.abs(xv).max()
    # s_t is amax / 2688 up to one binary32 rounding
    assert abs(float(s_t) * 2688.0 - amax_t) <= amax_t * 2.0 ** -23
    blocks = xv.reshape(128, 64, 16)
    ba = np.abs(blocks).max(axis=-1)
    sbv = np.vectorize(fpref.e4m3_value)(scales.astype(np.int64))
    target = ba / (6.0 * float(s_t))
    # block scale is the E4M3 value nearest the target (normal range: rel err <= 2^-4)
    normal = sbv >= 2.0 ** -6
    assert np.all(np.abs(sbv - target)[normal] <= target[normal] * 2.0 ** -4 * 1.0001)
    u = _unpack(codes, 1024).reshape(128, 64, 16)
    deq = fpref.E2M1_VALUES[u] * (sbv * float(s_t))[..., None]
    den = (sbv * float(s_t))[..., None]
    # every element within half an E2M1 step (<= 1 * den) of its value, blocks not saturating
    assert np.all(np.abs(deq - blocks)[normal] <= den.repeat(16, -1)[normal] * 1.0001 + 1e-30)
    # the block max maps to magnitude 6 (code 7) when sb is a normal E4M3 value
    imax = np.abs(blocks).argmax(axis=-1)
    top = np.take_along_axis(u & 7, imax[..., None], axis=-1)[..., 0]
    assert np.all(top[normal] == 7)


def test_nvfp4_zero_cases(oracle):
    z = np.zeros((4, 64), dtype=np.uint16)
    codes, scales, s_t = oracle.nvfp4_quantize(z)
    assert s_t == 0 and not codes.any() and not scales.any()
    x = synth.bf16_normal(4, 64, 1.0, seed=23)
    x[1, 16:32] = 0
    x[2, 32:48] = 0x8000
    codes, scales, s_t = oracle.nvfp4_quantize(x)
    u = _unpack(codes, 64)
    assert scales[1, 1] == 0 and not u[1, 16:32].any()
    assert scales[2, 2] == 0 and not u[2, 32:48].any()


# ----------------------------------------------------------------- bidimensional NVFP4

def _exact_regime_nvfp4(rows, cols, seed):
    """BF16 x whose rowwise NVFP4 quantize is exact (s_t = 2^-3, every block
    scale a power of two) with the expected codes from the nearest-grid
    search; see test_nvfp4_exact_regime_reduces_to_nearest_grid."""
    rng = np.random.default_rng(seed)
    p = -3
    q = rng.integers(-6, 3, size=(rows, cols // 16))
    blk_amax = 6.0 * 2.0 ** p * np.ldexp(1.0, q)
    x = rng.uniform(-1, 1, size=(rows, cols // 16, 16)) * blk_amax[..., None]
    x[..., 0] = blk_amax
    x = x.reshape(rows, cols)
    x[0, :16] = 0
    x[0, 0] = 2688.0 * 2.0 ** p
    xb = synth.f32_to_bf16_bits(x.astype(np.float32))
    blocks = fpref.bf16_bits_to_f64(xb).reshape(rows, cols // 16, 16)
    den = np.abs(blocks).max(axis=-1) / 6.0        # = E4M3(sb) * s_t, a power of two
    den[0, 0] = 2688.0 * 2.0 ** p / 6.0
    codes = fpref.nearest_e2m1_codes_vec(blocks / den[..., None]).reshape(rows, cols)
    return xb, codes


def test_nvfp4_quantize_2d_columnwise_exact_regime(oracle):
    """x is the transpose of an exact-regime matrix, so the columnwise output
    of x (the rowwise quantize of x^T) has codes fixed by the nearest-grid
    search, laid out [cols, rows/2]."""
    xt, expected = _exact_regime_nvfp4(96, 160, 31)
    x = np.ascontiguousarray(xt.T)                 # [160, 96]
    codes, scales, codes_t, scales_t, s_t = oracle.nvfp4_quantize_2d(x)
    assert s_t == np.float32(2.0 ** -3)
    assert codes.shape == (160, 48) and codes_t.shape == (96, 80)
    assert scales.shape == (160, 6) and scales_t.shape == (96, 10)
    assert np.array_equal(_unpack(codes_t, 160), expected)


def test_nvfp4_quantize_2d_orientation(oracle):
    """A large element at (0, 0) fixes s_t; one small element at (r, c) lands at
    row r, column c rowwise and at row c, column r columnwise."""
    r, c = 45, 70
    x = np.zeros((64, 96), dtype=np.uint16)
    x[0, 0] = synth.f32_to_bf16_bits(np.array([336.0], np.float32))[0]  # s_t = 336 / 2688 = 1/8
    x[r, c] = synth.f32_to_bf16_bits(np.array([-0.75], np.float32))[0]
    codes, scales, codes_t, scales_t, s_t = oracle.nvfp4_quantize_2d(x)
    assert s_t == np.float32(0.125)
    u, ut = _unpack(codes, 96), _unpack(codes_t, 64)
    # block amax 0.75: sb = E4M3(0.75 / 0.75) = 1.0 (byte 0x38), den = 1/8, -0.75 * 8 = -6 -> 15
    assert u[r, c] == 15 and ut[c, r] == 15
    assert scales[r, c // 16] == 0x38 and scales_t[c, r // 16] == 0x38
    assert np.count_nonzero(u) == 2 and np.count_nonzero(ut) == 2


def test_nvfp4_quantize_2d_symmetric_input(oracle):
    x = synth.bf16_normal(128, 128, 2.0, seed=32)
    x = np.triu(x) + np.triu(x, 1).T
    codes, scales, codes_t, scales_t, _ = oracle.nvfp4_quantize_2d(x)
    assert np.array_equal(codes, codes_t) and np.array_equal(scales, scales_t)
    # stochastic rounding: the same scales, but the two directions draw differently
    c2, s2, ct2, st2, _ = oracle.nvfp4_quantize_2d(x, seed=5)
    assert np.array_equal(s2, scales) and np.array_equal(st2, scales)
    assert not np.array_equal(c2, ct2)
