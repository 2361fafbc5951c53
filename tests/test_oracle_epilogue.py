"""Pins of the oracle's GEMM epilogue (bias, GELU, beta), CPU only.

GELU is checked against values fixed outside the oracle: the standard normal
CDF at 1 and 2 (Phi(1) = 0.8413447460685429, Phi(2) = 0.9772498680518208),
scipy's normal CDF, the identity GELU(-y) = GELU(y) - y (from
Phi(-y) = 1 - Phi(y)) and the limits GELU(y) -> y, GELU(-y) -> 0.  The bias,
beta and activation order against brute-force loops on tiny inputs.
"""
import math

import numpy as np
import pytest

import oracle


def test_gelu_known_values():
    assert oracle.gelu(0.0) == 0.0
    assert abs(oracle.gelu(1.0) - 0.8413447460685429) < 1e-15
    assert abs(oracle.gelu(-1.0) - (-0.15865525393145707)) < 1e-15
    assert abs(oracle.gelu(2.0) - 2 * 0.9772498680518208) < 1e-15
    assert oracle.gelu(40.0) == 40.0 and oracle.gelu(-40.0) == 0.0


def test_gelu_against_scipy_normal_cdf():
    stats = pytest.importorskip("scipy.stats")
    ys = np.linspace(-8, 8, 1001)
    ref = ys * stats.norm.cdf(ys)
    got = np.array([oracle.gelu(y) for y in ys])
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-300)   # a few ulps of the tail functions


def test_gelu_reflection_identity():
    rng = np.random.default_rng(2)
    for y in rng.uniform(-6, 6, 200):
        assert abs(oracle.gelu(-y) - (oracle.gelu(y) - y)) <= 4e-16 * max(1.0, abs(y))


def test_epilogue_terms_and_order():
    rng = np.random.default_rng(3)
    m, n = 3, 5
    d = rng.standard_normal((m, n))
    c = rng.standard_normal((m, n))
    bias = rng.standard_normal(n).astype(np.float32)
    beta = 0.75
    # identity: nothing added
    assert np.array_equal(oracle.gemm_epilogue(d), d)
    out = oracle.gemm_epilogue(d, bias=bias, gelu_on=True, beta=beta, c=c)
    for i in range(m):
        for j in range(n):
            y = d[i, j] + beta * c[i, j] + float(bias[j])     # bias per column, then GELU
            assert out[i, j] == 0.5 * y * math.erfc(-y / math.sqrt(2))
    # the bias is broadcast along rows (one value per output column)
    out = oracle.gemm_epilogue(np.zeros((m, n)), bias=bias)
    assert np.array_equal(out, np.tile(bias.astype(np.float64), (m, 1)))
    # beta alone is linear in c
    assert np.array_equal(oracle.gemm_epilogue(d, beta=2.0, c=c), d + 2.0 * c)
