"""The oracle's FP4 code transpose (oracle.fp4_transpose), pinned by what
defines it: the element at (r, c) of the FP4 matrix lands at (c, r), with the
nibble order of reading R2 (element 2t of a row in the low nibble of byte t);
the decoded values are the transpose of the decoded values; and transposing
twice gives the codes back.  "Integrate MXFP4 hipblaslt GEMM support",
Takeaways: the layouts other than TN come down to this transpose of one
operand."""
import numpy as np
import pytest

import oracle


def _nibble(codes, rows, cols, r, c):
    """Code of element (r, c) read straight from the packed bytes."""
    byte = int(codes.reshape(rows, cols // 2)[r, c // 2])
    return (byte >> 4) if c % 2 else (byte & 0xF)


@pytest.mark.parametrize("rows,cols", [(2, 2), (4, 6), (32, 64), (6, 32)])
def test_each_element_moves_to_the_transposed_position(rows, cols):
    rng = np.random.default_rng(rows * 100 + cols)
    codes = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    t = oracle.fp4_transpose(codes, rows, cols)
    assert t.shape == (cols, rows // 2) and t.dtype == np.uint8
    for r in range(rows):
        for c in range(cols):
            assert _nibble(t, cols, rows, c, r) == _nibble(codes, rows, cols, r, c), (r, c)


def test_single_code_probe():
    # one nonzero code at (r, c) = (5, 2) of a 6 x 8 matrix: byte 1 of row 5,
    # low nibble; transposed it is element (2, 5): byte 2 of row 2, high nibble
    codes = np.zeros((6, 4), np.uint8)
    codes[5, 1] = 0x07
    t = oracle.fp4_transpose(codes, 6, 8)
    expect = np.zeros((8, 3), np.uint8)
    expect[2, 2] = 0x70
    assert np.array_equal(t, expect)


def test_decoded_values_transpose_and_twice_is_identity():
    rows, cols = 64, 96
    rng = np.random.default_rng(7)
    codes = rng.integers(0, 256, size=(rows, cols // 2), dtype=np.uint8)
    t = oracle.fp4_transpose(codes, rows, cols)
    assert np.array_equal(oracle.e2m1_decode_array(t, rows),
                          oracle.e2m1_decode_array(codes, cols).T)
    assert np.array_equal(oracle.fp4_transpose(t, cols, rows), codes)


def test_gemm_of_transposed_operand_is_the_nn_product():
    # A stored K x M (M contiguous) is the NN operand; transposed to M x K it
    # gives, through the TN definition, D = A B^T computed from the values
    m, n, k = 32, 32, 64
    rng = np.random.default_rng(11)
    a_mn = rng.integers(0, 256, size=(k, m // 2), dtype=np.uint8)   # [K, M/2]
    b = rng.integers(0, 256, size=(n, k // 2), dtype=np.uint8)
    sa = rng.integers(124, 131, size=(m, k // 32), dtype=np.uint8)
    sb = rng.integers(124, 131, size=(n, k // 32), dtype=np.uint8)
    a_km = oracle.fp4_transpose(a_mn, k, m)                          # [M, K/2]
    d, _ = oracle.mx_gemm(a_km, sa, b, sb, m, n, k)
    av = oracle.e2m1_decode_array(a_mn, m).T * np.repeat(2.0 ** (sa.astype(np.float64) - 127), 32, axis=1)
    bv = oracle.e2m1_decode_array(b, k) * np.repeat(2.0 ** (sb.astype(np.float64) - 127), 32, axis=1)
    assert np.all(np.abs(d - av @ bv.T) <= 1e-12 * (np.abs(av) @ np.abs(bv).T))
