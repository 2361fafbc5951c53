"""Pins of the oracle's element and scale codecs (CPU only).

Each check compares the oracle with something other than itself: the
formats' bit-field definitions, exact-rational brute force, Python's frexp,
and torch's BF16 / float8_e4m3fn conversions.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

from tests import fpref


def test_e2m1_decode_matches_bitfield_definition(oracle):
    for c in range(16):
        assert oracle.e2m1_decode(c) == fpref.e2m1_value(c)
    # the OCP E2M1 magnitude set
    assert sorted({abs(fpref.e2m1_value(c)) for c in range(16)}) == [0, .5, 1, 1.5, 2, 3, 4, 6]


def test_e2m1_round_trip_all_16_codes(oracle):
    for c in range(16):
        assert oracle.e2m1_encode(oracle.e2m1_decode(c)) == c


@pytest.mark.parametrize("y,code", [
    # ties go to the even code (mantissa bit 0)
    (0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
    # just off the ties
    (0.2500001, 1), (0.7499999, 1), (1.2500001, 3), (4.9999, 6), (5.0001, 7),
    # saturation
    (6.0, 7), (6.9, 7), (7.0, 7), (1e30, 7),
    # signs, including values that round to zero
    (-0.1, 8), (-0.0, 8), (0.0, 0), (-5.5, 15), (-0.75, 10),
])
def test_e2m1_encode_closed_forms(oracle, y, code):
    assert oracle.e2m1_encode(y) == code


def test_e2m1_encode_brute_force_dense(oracle):
    # every multiple of 1/64 in [-8, 8] plus the BF16 values in that range
    ys = [i / 64 for i in range(-512, 513)]
    rng = np.random.default_rng(1)
    ys += list(rng.uniform(-9, 9, 2000))
    for y in ys:
        assert oracle.e2m1_encode(y) == fpref.nearest_e2m1_code(y), y


def test_bf16_decode_matches_torch_exhaustive(oracle):
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    got = np.array([oracle.bf16_to_float(int(b)) for b in bits], dtype=np.float32)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite].view(np.uint32), ref[finite].view(np.uint32))


def test_bf16_floor_log2_matches_frexp_exhaustive(oracle):
    for b in range(65536):
        e = (b >> 7) & 0xFF
        if e == 0xFF or (b & 0x7FFF) == 0:
            continue
        v = float(fpref.bf16_bits_to_f64(np.array([b], np.uint16))[0])
        assert oracle.bf16_floor_log2(b) == math.frexp(abs(v))[1] - 1, hex(b)


def test_ue8m0_decode(oracle):
    for e in range(255):
        assert oracle.ue8m0_decode(e) == fpref.ue8m0_value(e)
    assert oracle.ue8m0_decode(127) == 1.0
    assert oracle.ue8m0_decode(128) == 2.0


def test_e4m3_decode_matches_torch_and_fields(oracle):
    for b in range(256):
        if (b & 0x7F) == 0x7F:
            continue  # NaN
        ref = torch.tensor([b], dtype=torch.uint8).view(torch.float8_e4m3fn).double().item()
        assert oracle.e4m3_decode(b) == ref == fpref.e4m3_value(b)
    assert oracle.e4m3_decode(0x7E) == 448.0
    assert oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch(oracle):
    rng = np.random.default_rng(2)
    vals = np.concatenate([
        rng.uniform(0, 463.9, 4000), np.exp(rng.uniform(-12, 6, 4000)),
        np.array([oracle.e4m3_decode(c) for c in range(0x7F)]),
    ]).astype(np.float32)
    # midpoints between neighbouring codes (exact ties)
    grid = [oracle.e4m3_decode(c) for c in range(0x7F)]
    mids = np.array([(grid[i] + grid[i + 1]) / 2 for i in range(len(grid) - 1)], np.float32)
    vals = np.concatenate([vals, mids])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for v, r in zip(vals.tolist(), ref.tolist()):
        assert oracle.e4m3_encode(v) == r, v


def test_e4m3_encode_ties_and_saturation(oracle):
    for c in range(0x7E):
        lo, hi = oracle.e4m3_decode(c), oracle.e4m3_decode(c + 1)
        mid = (lo + hi) / 2
        assert oracle.e4m3_encode(mid) == (c if c % 2 == 0 else c + 1)
        assert oracle.e4m3_encode(lo) == c
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(1000.0) == 0x7E
    assert oracle.e4m3_encode(0.0) == 0
    assert oracle.e4m3_encode(2.0 ** -10) == 0       # tie with 0 -> even (0)
    assert oracle.e4m3_encode(2.0 ** -10 * 1.01) == 1


def _nearest_bf16_bits(x: float) -> int:
    """Exact-rational brute force over the BF16 neighbours of x (ties to even)."""
    f = Fraction(x)
    # candidates: BF16 values around x, found by scanning the bit patterns near
    # the truncation of x's binary32 image
    t = np.array([x], dtype=np.float32).view(np.uint32)[0] >> 16
    best = None
    for b in range(max(0, int(t) - 2), min(0xFFFF, int(t) + 3)):
        if ((b >> 7) & 0xFF) == 0xFF:
            continue
        v = Fraction(float(fpref.bf16_bits_to_f64(np.array([b], np.uint16))[0]))
        d = abs(f - v)
        if best is None or d < best[0] or (d == best[0] and b % 2 == 0):
            best = (d, b)
    return best[1]


def test_round_bf16_brute_force(oracle):
    rng = np.random.default_rng(3)
    xs = list(rng.standard_normal(3000) * np.exp(rng.uniform(-30, 30, 3000)))
    xs += [1 + 2 ** -8, 1 + 3 * 2 ** -8, 1 + 2 ** -8 + 2 ** -30, 1 + 2 ** -8 - 2 ** -40,
           2.0 ** -130 * 1.5, 2.0 ** -133, 2.0 ** -134 * 3]
    got = oracle.round_bf16(np.array(xs))
    for x, g in zip(xs, got.tolist()):
        ref = _nearest_bf16_bits(abs(x)) | (0x8000 if x < 0 else 0)
        assert g == ref, x
    # a value just above a BF16 midpoint must not be rounded twice
    assert oracle.round_bf16(np.array([1 + 2 ** -8 + 2 ** -30]))[0] == 0x3F81
    assert oracle.round_bf16(np.array([1 + 2 ** -8]))[0] == 0x3F80
