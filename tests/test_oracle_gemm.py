"""Pins of the oracle's block-scaled GEMM (CPU only)."""
import numpy as np
import pytest

from block_scaled_fp4_bf16_gb300 import synth
from tests import fpref


def _dequant(codes, scales, k, blk, scale_fn):
    v = fpref.decode_fp4_matrix(codes, k)
    s = np.vectorize(scale_fn, otypes=[np.float64])(scales.astype(np.int64))
    return v * np.repeat(s, blk, axis=1)


@pytest.mark.parametrize("m,n,k", [(32, 32, 256), (64, 32, 512), (32, 64, 256), (64, 64, 512)])
def test_mx_gemm_equals_dequantize_then_fp64_matmul(oracle, m, n, k):
    """Brute force: CPU-dequantize both operands, numpy fp64 matmul.  With
    scale exponents in [120, 134] every partial sum is exact in binary64, so
    the two must agree bit for bit."""
    rng = np.random.default_rng(m * 7 + n * 3 + k)
    a = rng.integers(0, 256, size=(m, k // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sa = rng.integers(120, 135, size=(m, k // 32), dtype=np.uint8)
    sb = rng.integers(120, 135, size=(n, k // 32), dtype=np.uint8)
    d, s_abs = oracle.mx_gemm(a, sa, b, sb, m, n, k)
    A = _dequant(a, sa, k, 32, fpref.ue8m0_value)
    B = _dequant(b, sb, k, 32, fpref.ue8m0_value)
    assert np.array_equal(d, A @ B.T)
    assert np.array_equal(s_abs, np.abs(A) @ np.abs(B).T)


def test_nvfp4_gemm_equals_dequantize_then_fp64_matmul(oracle):
    rng = np.random.default_rng(5)
    m, n, k = 32, 64, 256
    a = rng.integers(0, 256, size=(m, k // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sa = rng.integers(0, 0x7F, size=(m, k // 16), dtype=np.uint8)
    sb = rng.integers(0, 0x7F, size=(n, k // 16), dtype=np.uint8)
    ta, tb = np.float32(0.375), np.float32(1.25e-3)
    d, s_abs = oracle.nvfp4_gemm(a, sa, b, sb, m, n, k, ta, tb)
    A = _dequant(a, sa, k, 16, fpref.e4m3_value)
    B = _dequant(b, sb, k, 16, fpref.e4m3_value)
    ref = (A @ B.T) * (float(ta) * float(tb))
    np.testing.assert_allclose(d, ref, rtol=1e-14, atol=1e-300)


def test_all_ones_gives_k(oracle):
    for m, n, k in [(32, 32, 256), (64, 96, 1024)]:
        a = np.full((m, k // 2), 0x22, np.uint8)     # both nibbles code 2 = 1.0
        b = np.full((n, k // 2), 0x22, np.uint8)
        s = lambda r: np.full((r, k // 32), 127, np.uint8)
        d, _ = oracle.mx_gemm(a, s(m), b, s(n), m, n, k)
        assert np.all(d == k)


def test_scale_exponent_plus_one_doubles_block_term(oracle):
    rng = np.random.default_rng(6)
    m, n, k = 32, 32, 512
    a = rng.integers(0, 256, size=(m, k // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sa = rng.integers(122, 131, size=(m, k // 32), dtype=np.uint8)
    sb = rng.integers(122, 131, size=(n, k // 32), dtype=np.uint8)
    d0, _ = oracle.mx_gemm(a, sa, b, sb, m, n, k)
    j = 5
    # contribution of block j alone
    a_only = np.zeros_like(a)
    a_only[:, j * 16:(j + 1) * 16] = a[:, j * 16:(j + 1) * 16]
    dj, _ = oracle.mx_gemm(a_only, sa, b, sb, m, n, k)
    sa2 = sa.copy()
    sa2[:, j] += 1
    d1, _ = oracle.mx_gemm(a, sa2, b, sb, m, n, k)
    assert np.array_equal(d1 - d0, dj)


def test_sign_flip_negates(oracle):
    rng = np.random.default_rng(7)
    m, n, k = 32, 64, 256
    a = rng.integers(0, 256, size=(m, k // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sa = rng.integers(120, 135, size=(m, k // 32), dtype=np.uint8)
    sb = rng.integers(120, 135, size=(n, k // 32), dtype=np.uint8)
    d, s_abs = oracle.mx_gemm(a, sa, b, sb, m, n, k)
    dn, s_abs_n = oracle.mx_gemm(a ^ 0x88, sa, b, sb, m, n, k)
    assert np.array_equal(dn, -d)
    assert np.array_equal(s_abs_n, s_abs)
    # transposition symmetry
    dt, _ = oracle.mx_gemm(b, sb, a, sa, n, m, k)
    assert np.array_equal(dt, d.T)
    # s_abs is the GEMM of the magnitudes
    dabs, _ = oracle.mx_gemm(a & 0x77, sa, b & 0x77, sb, m, n, k)
    assert np.array_equal(dabs, s_abs)


def test_row_col_sampling_matches_full(oracle):
    rng = np.random.default_rng(8)
    m, n, k = 96, 64, 512
    a = rng.integers(0, 256, size=(m, k // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sa = rng.integers(120, 135, size=(m, k // 32), dtype=np.uint8)
    sb = rng.integers(120, 135, size=(n, k // 32), dtype=np.uint8)
    d, s = oracle.mx_gemm(a, sa, b, sb, m, n, k)
    rows = np.array([0, 7, 95, 33])
    cols = np.array([63, 0, 12])
    d2, s2 = oracle.mx_gemm(a, sa, b, sb, m, n, k, rows=rows, cols=cols)
    assert np.array_equal(d2, d[np.ix_(rows, cols)])
    assert np.array_equal(s2, s[np.ix_(rows, cols)])


def test_nvfp4_reduces_to_mx_with_power_of_two_scales(oracle):
    """When every E4M3 block scale and both tensor scales are powers of two, the
    NVFP4 GEMM is the MX GEMM with the equivalent UE8M0 exponents."""
    rng = np.random.default_rng(9)
    m, n, k = 32, 32, 512
    a = rng.integers(0, 256, size=(m, k // 2), dtype=np.uint8)
    b = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    ea = rng.integers(-4, 5, size=(m, k // 32))
    eb = rng.integers(-4, 5, size=(n, k // 32))
    # E4M3 byte of 2^e (normal): exponent field e + 7, mantissa 0
    to_e4m3 = lambda e: ((e + 7) << 3).astype(np.uint8)
    sa_nv = np.repeat(to_e4m3(ea), 2, axis=1)   # two 16-blocks per 32-block
    sb_nv = np.repeat(to_e4m3(eb), 2, axis=1)
    ta, tb = np.float32(2.0 ** -3), np.float32(2.0 ** 5)
    d_nv, _ = oracle.nvfp4_gemm(a, sa_nv, b, sb_nv, m, n, k, ta, tb)
    d_mx, _ = oracle.mx_gemm(a, (ea + 127).astype(np.uint8), b, (eb + 127).astype(np.uint8), m, n, k)
    assert np.array_equal(d_nv, d_mx * 2.0 ** 2)


def test_scale_tile_is_a_padded_permutation(oracle):
    rng = np.random.default_rng(10)
    for rows, kb in [(128, 8), (32, 8), (200, 16), (256, 4)]:
        plain = rng.integers(1, 256, size=(rows, kb), dtype=np.uint8)
        t = oracle.scale_tile(plain)
        rows_pad = (rows + 127) // 128 * 128
        assert t.size == rows_pad * kb
        assert np.array_equal(np.sort(t[t != 0]), np.sort(plain.ravel()))
        assert np.count_nonzero(t) == rows * kb
        # spot positions of the documented 128x4 atom
        atoms_k = kb // 4
        assert t[0] == plain[0, 0]
        assert t[1] == plain[0, 1]
        assert t[16] == plain[1, 0]
        if rows > 32:
            assert t[4] == plain[32, 0]
        if kb > 4:
            assert t[512] == plain[0, 4]
        if rows > 128:
            assert t[atoms_k * 512] == plain[128, 0]
