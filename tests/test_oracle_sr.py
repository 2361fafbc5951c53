"""Pins of the oracle's stochastic-rounding path (NVFP4), CPU only.

What fixes each piece independently of the oracle's own code:
  * Philox4x32: the known-answer vectors published with the generator
    (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2,
    3", SC 2011; the Random123 distribution's known-answer tests for
    philox4x32 at 7 and 10 rounds).
  * the element rounding: exact rational arithmetic (fractions.Fraction)
    over a brute-force search of the E2M1 grid, and the probability statement
    that defines stochastic rounding (the number of bytes u that round up is
    ceil(256 p)).
  * the quantizer: its scales and s_t are the round-to-nearest quantizer's;
    every code is one of the two grid neighbours of x / den; inputs built so
    that every quotient sits exactly half-way between two neighbours expose
    which byte of which draw each element used; and the mean over many seeds
    converges to x / den (unbiasedness).
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle

GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]

# (rounds, counter, key, expected) -- the published philox4x32 known answers
KAT = [
    (7, [0, 0, 0, 0], [0, 0], [0x5F6FB709, 0x0D893F64, 0x4F121F81, 0x4F730A48]),
    (7, [0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x5207DDC2, 0x45165E59, 0x4D8EE751, 0x8C52F662]),
    (7, [0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
     [0x4DFCCABA, 0x190A87F0, 0xC47362BA, 0xB6B5242A]),
    (10, [0, 0, 0, 0], [0, 0], [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]),
    (10, [0xFFFFFFFF] * 4, [0xFFFFFFFF] * 2, [0x408F276D, 0x41C83B0E, 0xA20BC7C6, 0x6D5451FD]),
    (10, [0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344], [0xA4093822, 0x299F31D0],
     [0xD16CFE09, 0x94FDCCEB, 0x5001E420, 0x24126EA1]),
]


@pytest.mark.parametrize("rounds,ctr,key,want", KAT)
def test_philox_known_answers(rounds, ctr, key, want):
    assert [int(v) for v in oracle.philox4x32(ctr, key, rounds)] == want


def test_philox_zero_rounds_is_identity():
    ctr = [1, 2, 3, 4]
    assert [int(v) for v in oracle.philox4x32(ctr, [5, 6], 0)] == ctr


def test_philox_rounds_compose_with_bumped_key():
    """R rounds = 1 round, then R-1 rounds under the key bumped once."""
    rng = np.random.default_rng(11)
    for _ in range(20):
        ctr = rng.integers(0, 2**32, 4, dtype=np.uint64).astype(np.uint32)
        key = rng.integers(0, 2**32, 2, dtype=np.uint64).astype(np.uint32)
        one = oracle.philox4x32(ctr, key, 1)
        bumped = [(int(key[0]) + 0x9E3779B9) & 0xFFFFFFFF, (int(key[1]) + 0xBB67AE85) & 0xFFFFFFFF]
        assert np.array_equal(oracle.philox4x32(one, bumped, 9), oracle.philox4x32(ctr, key, 10))


def _sr_reference(y: float, u: int) -> int:
    """Exact-rational stochastic rounding of y to an E2M1 code."""
    a = abs(Fraction(y))
    sign = 8 if np.signbit(y) else 0
    if a >= 6:
        return 7 | sign
    lo = max(i for i, g in enumerate(GRID) if Fraction(g) <= a)
    p = (a - Fraction(GRID[lo])) / (Fraction(GRID[lo + 1]) - Fraction(GRID[lo]))
    return (lo + 1 if Fraction(u, 256) < p else lo) | sign


def test_sr_encode_matches_exact_rationals():
    rng = np.random.default_rng(5)
    ys = rng.uniform(-7.0, 7.0, 300).astype(np.float32)
    ys = np.concatenate([ys, np.float32(GRID), -np.float32(GRID), np.float32([0.25, 1.25, 5.0, 6.5, 1e-30, -1e-30])])
    for y in ys:
        for u in range(0, 256, 5):
            assert oracle.e2m1_encode_sr(float(y), u) == _sr_reference(float(y), u), (float(y), u)


def test_sr_encode_probability_is_ceil_256p():
    """Exactly ceil(256 p) of the 256 byte values round up; all of them are 0..255 monotone."""
    rng = np.random.default_rng(6)
    for y in rng.uniform(0.0, 5.999, 200).astype(np.float32):
        a = Fraction(float(y))
        lo = max(i for i, g in enumerate(GRID) if Fraction(g) <= a)
        p = (a - Fraction(GRID[lo])) / (Fraction(GRID[lo + 1]) - Fraction(GRID[lo]))
        ups = [oracle.e2m1_encode_sr(float(y), u) == lo + 1 for u in range(256)]
        downs = [oracle.e2m1_encode_sr(float(y), u) == lo for u in range(256)]
        assert all(x or d for x, d in zip(ups, downs))
        n_up = sum(ups)
        assert n_up == -(-p.numerator * 256 // p.denominator)  # ceil(256 p)
        assert ups == [True] * n_up + [False] * (256 - n_up)  # the smallest bytes round up


def test_sr_encode_grid_points_and_saturation():
    for u in range(256):
        for c, g in enumerate(GRID):
            assert oracle.e2m1_encode_sr(g, u) == c
            assert oracle.e2m1_encode_sr(-g, u) == c | 8
        assert oracle.e2m1_encode_sr(6.25, u) == 7
        assert oracle.e2m1_encode_sr(-100.0, u) == 15


def _bf16(v):
    f = np.asarray(v, dtype=np.float32)
    bits = f.view(np.uint32)
    assert np.all(bits & 0xFFFF == 0), "test values must be exact BF16"
    return (bits >> 16).astype(np.uint16)


def _random_bf16(rows, cols, seed):
    rng = np.random.default_rng(seed)
    f = (rng.standard_normal((rows, cols)) * 0.02).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def _decode(codes):
    lo = codes & 0xF
    hi = codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(codes.shape[0], -1)
    mag = np.float64(GRID)[c & 7]
    return np.where(c & 8, -mag, mag), c


def _e4m3_values(scales):
    return np.array([oracle.e4m3_decode(int(b)) for b in range(256)])[scales]


def test_sr_scales_equal_round_to_nearest_and_codes_are_neighbours():
    x = _random_bf16(48, 96, 1)
    x[3, :16] = 0  # an all-zero block
    rc, rs, rt = oracle.nvfp4_quantize(x)
    for seed in (0, 1, 0xDEADBEEF12345678):
        sc, ss, st = oracle.nvfp4_quantize_sr(x, seed)
        assert np.array_equal(ss, rs) and st == rt
        xv = (x.astype(np.uint32) << 16).view(np.float32)
        den = np.repeat((_e4m3_values(ss) * np.float64(st)).astype(np.float32), 16, axis=1)
        q = np.abs(np.where(den > 0, xv / np.where(den > 0, den, 1), 0)).astype(np.float64)
        mag, c = _decode(sc)
        lo = np.array([[max(i for i, g in enumerate(GRID) if g <= min(v, 6.0)) for v in row] for row in q])
        assert np.all(((c & 7) == lo) | ((c & 7) == np.minimum(lo + 1, 7)))
        assert np.all(sc[3, :8] == 0)
        # the round-to-nearest code is one of the two as well
        _, cr = _decode(rc)
        assert np.all(np.abs((cr & 7).astype(int) - (c & 7).astype(int)) <= 1)


def _halfway_input(rows, nblocks):
    """BF16 [rows, 16 * (nblocks + 1)]: block 0 of every row holds 10.5 (so
    amax = 10.5 and s_t = 10.5 / 2688 = 2^-8); every other block holds 6.0
    (sb = E4M3(6 / (6 * 2^-8)) = 256, den = 1) and fifteen values exactly
    half-way between two E2M1 neighbours, so p = 1/2 for each of them."""
    halves = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    rng = np.random.default_rng(3)
    f = np.zeros((rows, 16 * (nblocks + 1)), dtype=np.float32)
    f[:, 0] = 10.5
    for r in range(rows):
        for b in range(1, nblocks + 1):
            v = rng.choice(halves, 16) * rng.choice([-1.0, 1.0], 16)
            v[int(rng.integers(0, 16))] = 6.0
            f[r, 16 * b:16 * (b + 1)] = v
    return f, _bf16(f)


@pytest.mark.parametrize("seed,rounds", [(0, 10), (0x0123456789ABCDEF, 10), (77, 7)])
def test_sr_draw_layout_exposed_by_halfway_values(seed, rounds):
    """Element i of block (r, j) rounds up iff byte i of the draw of counter
    (j, r, 0, 0) under key (seed low, seed high) is below 128."""
    rows, nblocks = 5, 6
    f, x = _halfway_input(rows, nblocks)
    codes, scales, st = oracle.nvfp4_quantize_sr(x, seed, rounds)
    assert st == np.float32(2.0 ** -8)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    _, c = _decode(codes)
    for r in range(rows):
        for j in range(1, nblocks + 1):
            assert scales[r, j] == 0x78  # E4M3 256 = 2^8 (exponent 15, mantissa 0)
            draw = oracle.philox4x32([j, r, 0, 0], key, rounds)
            for i in range(16):
                v = abs(float(f[r, 16 * j + i]))
                if v == 6.0:
                    assert c[r, 16 * j + i] & 7 == 7
                    continue
                u = (int(draw[i // 4]) >> (8 * (i % 4))) & 0xFF
                lo = max(k for k, g in enumerate(GRID) if g <= v)
                assert c[r, 16 * j + i] & 7 == (lo + 1 if u < 128 else lo), (r, j, i)


def test_sr_direction_and_seed_change_the_draws():
    x = _random_bf16(32, 64, 2)
    a = oracle.nvfp4_quantize_sr(x, 9)[0]
    assert np.array_equal(a, oracle.nvfp4_quantize_sr(x, 9)[0])  # deterministic
    assert not np.array_equal(a, oracle.nvfp4_quantize_sr(x, 10)[0])
    assert not np.array_equal(a, oracle.nvfp4_quantize_sr(x, 9, direction=1)[0])
    assert not np.array_equal(a, oracle.nvfp4_quantize_sr(x, 9, rounds=7)[0])
    assert not np.array_equal(a, oracle.nvfp4_quantize_sr(x, 9 | (1 << 40))[0])


def test_sr_is_unbiased_over_seeds():
    """The mean of the dequantized codes over many seeds approaches x / den.

    Per element the expectation is lo + step * ceil(256 p) / 256, within
    step / 256 of x / den; the standard error of a mean of 400 draws is at
    most step / 40, so 5 standard errors plus the bias bound the error."""
    x = _random_bf16(4, 64, 4)
    _, scales, st = oracle.nvfp4_quantize(x)
    xv = (x.astype(np.uint32) << 16).view(np.float32)
    den = np.repeat((_e4m3_values(scales) * np.float64(st)).astype(np.float32), 16, axis=1)
    q = (xv / den).astype(np.float64)
    acc = np.zeros_like(q)
    n = 400
    for seed in range(n):
        acc += _decode(oracle.nvfp4_quantize_sr(x, 1000 + seed)[0])[0]
    mean = acc / n
    step = np.where(np.abs(q) < 2, 0.5, np.where(np.abs(q) < 4, 1.0, 2.0))
    assert np.all(np.abs(mean - q) <= step * (5 / 40 + 1 / 256))
    # and the spread is that of two-point rounding, not of round-to-nearest
    rne = _decode(oracle.nvfp4_quantize(x)[0])[0]
    assert np.mean(np.abs(mean - q)) < 0.5 * np.mean(np.abs(rne - q))


def test_sr_columnwise_draws_use_direction_one():
    """The columnwise output of the bidimensional quantize draws with direction
    1: with x the transpose of the half-way input, element i of columnwise block
    (r, j) rounds up iff byte i of the draw of counter (j, r, 1, 0) is < 128."""
    rows, nblocks, seed = 16, 3, 0xABCDEF0123
    f, xr = _halfway_input(rows, nblocks)
    x = np.ascontiguousarray(xr.T)                # [16 (nblocks + 1), 16]
    _, _, codes_t, scales_t, st = oracle.nvfp4_quantize_2d(x, seed=seed)
    assert st == np.float32(2.0 ** -8)
    _, c = _decode(codes_t)
    key = [seed & 0xFFFFFFFF, seed >> 32]
    for r in range(rows):
        for j in range(1, nblocks + 1):
            draw = oracle.philox4x32([j, r, 1, 0], key)
            for i in range(16):
                v = abs(float(f[r, 16 * j + i]))
                if v == 6.0:
                    continue
                u = (int(draw[i // 4]) >> (8 * (i % 4))) & 0xFF
                lo = max(k for k, g in enumerate(GRID) if g <= v)
                assert c[r, 16 * j + i] & 7 == (lo + 1 if u < 128 else lo)
