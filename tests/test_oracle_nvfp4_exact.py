"""Pin of the oracle's NVFP4 arithmetic: the binary32 operation order, restated
in exact rationals, CPU only.

NVIDIA/TransformerEngine #3809 (CuTeDSL NVFP4 quantize kernels), commit
messages: NVFP4 = E2M1 codes with E4M3 scales per 16 elements and an FP32
per-tensor amax, and round-to-nearest output is byte-identical across
implementations; configs name the tensor scale amax / (6 * 448).  The reading
the oracle implements is a fixed chain of binary32 round-to-nearest-even
operations:

    s_t   = RN(amax_t / 2688)
    t     = RN(6 * s_t)
    sb    = E4M3_RNE_satfinite(RN(amax_b / t))
    den   = RN(E4M3(sb) * s_t)
    q_i   = RN(x_i / den)
    code  = E2M1_RNE_sat(q_i)          (stochastic: the SR rule on q_i)

Here every one of those steps is computed from scratch with
fractions.Fraction, and each rounding to binary32 is a brute-force choice
between the two representable neighbours of the exact value (ties to the
even significand), with no float arithmetic of the machine involved.  The
E4M3 and E2M1 roundings are nearest-value searches over grids built from the
formats' bit fields, and Philox4x32 is restated in Python and checked
against its published known answers.

The inputs are chosen so that plausible slips in the oracle fail: random
tensors whose s_t and block scales are not powers of two, and adversarial
tensors whose quotients x / den, or whose block ratios amax_b / t, sit
within one binary32 ulp of an E2M1 or E4M3 rounding midpoint, or exactly
on one.  There, a reciprocal multiply x * RN(1 / den), the order
amax_b / 6 / s_t, a fused multiply-add, or a quotient rounded straight from
binary64 to E2M1 (skipping the binary32 rounding) each change bytes.
"""
from fractions import Fraction

import numpy as np
import pytest

from block_scaled_fp4_bf16_gb300 import synth

# ----------------------------------------------------------------- exact formats

E2M1_MAGS = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2), Fraction(2), Fraction(3),
             Fraction(4), Fraction(6)]


def _e4m3_from_fields(code: int) -> Fraction:
    """Non-negative E4M3 (bias 7, 3 mantissa bits, subnormals at exponent 0)."""
    e, m = (code >> 3) & 0xF, code & 7
    if e == 0:
        return Fraction(m, 8) * Fraction(1, 2 ** 6)
    return (1 + Fraction(m, 8)) * (Fraction(2) ** (e - 7))


E4M3_GRID = [_e4m3_from_fields(c) for c in range(0x7F)]   # 0x7F is NaN
E4M3_MAX = E4M3_GRID[0x7E]                                 # 448


def bf16_exact(bits: int) -> Fraction:
    """A BF16 bit pattern as an exact rational (sign, 8-bit exponent, 7-bit mantissa)."""
    s, e, m = (bits >> 15) & 1, (bits >> 7) & 0xFF, bits & 0x7F
    assert e != 0xFF, "Inf/NaN inputs are outside the contract"
    v = Fraction(m, 128) * Fraction(2) ** -126 if e == 0 else \
        (1 + Fraction(m, 128)) * Fraction(2) ** (e - 127)
    return -v if s else v


def rn_binary32(q: Fraction) -> Fraction:
    """q rounded to the nearest binary32 value, ties to the even significand."""
    if q == 0:
        return Fraction(0)
    neg = q < 0
    a = -q if neg else q
    n, d = a.numerator, a.denominator
    e = n.bit_length() - d.bit_length()
    if (n << max(0, -e)) < (d << max(0, e)):
        e -= 1                                   # now 2^e <= a < 2^(e+1)
    e = max(e, -126)                             # subnormals share the quantum 2^-149
    sh = e - 23                                  # the quantum is 2^sh
    num, den = (n, d << sh) if sh >= 0 else (n << -sh, d)
    lo, rem = divmod(num, den)                   # a / 2^sh lies in [lo, lo + 1)
    if 2 * rem > den or (2 * rem == den and lo & 1):
        lo += 1                                  # the nearer neighbour; even on a tie
    r = lo * Fraction(2) ** sh
    assert r < Fraction(2) ** 128, "binary32 overflow"
    return -r if neg else r


def e4m3_rne_satfinite(r: Fraction) -> int:
    """Nearest E4M3 code of r >= 0 (ties to the even code); r >= 448 gives 448."""
    assert r >= 0
    if r >= E4M3_MAX:
        return 0x7E
    best = 0
    for c in range(1, 0x7F):
        dc, db = abs(r - E4M3_GRID[c]), abs(r - E4M3_GRID[best])
        if dc < db or (dc == db and c % 2 == 0):
            best = c
    return best


def e2m1_rne(mag: Fraction, negative: bool) -> int:
    """Nearest E2M1 code of a magnitude (ties to the even code, saturating at 6),
    sign bit 3 set for a negative input even when the magnitude rounds to 0."""
    sign = 8 if negative else 0
    if mag >= 6:
        return 7 | sign
    best = 0
    for c in range(1, 8):
        dc, db = abs(mag - E2M1_MAGS[c]), abs(mag - E2M1_MAGS[best])
        if dc < db or (dc == db and c % 2 == 0):
            best = c
    return best | sign


def e2m1_sr(mag: Fraction, negative: bool, u: int) -> int:
    """Stochastic rounding with the byte u: lo <= mag < hi, p = (mag - lo) / (hi - lo);
    the magnitude is hi iff u / 256 < p; mag >= 6 saturates; the sign is kept."""
    sign = 8 if negative else 0
    if mag >= 6:
        return 7 | sign
    c = max(i for i in range(8) if E2M1_MAGS[i] <= mag)
    p = (mag - E2M1_MAGS[c]) / (E2M1_MAGS[c + 1] - E2M1_MAGS[c])
    return (c + 1 if Fraction(u, 256) < p else c) | sign


# ----------------------------------------------------------------- Philox4x32

M32 = 0xFFFFFFFF


def philox4x32(ctr, key, rounds):
    """Philox4x32-R (Salmon, Moraes, Dror, Shaw, SC 2011, Philox section)."""
    c0, c1, c2, c3 = (int(v) & M32 for v in ctr)
    k0, k1 = (int(v) & M32 for v in key)
    for i in range(rounds):
        if i:
            k0, k1 = (k0 + 0x9E3779B9) & M32, (k1 + 0xBB67AE85) & M32
        p0, p1 = 0xD2511F53 * c0, 0xCD9E8D57 * c2
        c0, c1, c2, c3 = ((p1 >> 32) ^ c1 ^ k0) & M32, p1 & M32, ((p0 >> 32) ^ c3 ^ k1) & M32, \
            p0 & M32
    return [c0, c1, c2, c3]


def test_python_philox_published_known_answers():
    # Random123 known-answer vectors for philox4x32 (7 and 10 rounds)
    assert philox4x32([0] * 4, [0, 0], 10) == [0x6627E8D5, 0xE169C58D, 0xBC57AC4C, 0x9B00DBD8]
    assert philox4x32([M32] * 4, [M32] * 2, 7) == [0x5207DDC2, 0x45165E59, 0x4D8EE751,
                                                    0x8C52F662]
    assert philox4x32([0x243F6A88, 0x85A308D3, 0x13198A2E, 0x03707344],
                      [0xA4093822, 0x299F31D0], 10) == [0xD16CFE09, 0x94FDCCEB, 0x5001E420,
                                                       0x24126EA1]


# ----------------------------------------------------------------- the restatement

def nvfp4_exact(x_bits, seed=None, rounds=10, direction=0):
    """NVFP4 quantize of BF16 bits [rows, cols] in exact rationals.

    Returns (codes [rows, cols/2] with element 2t in the low nibble, E4M3
    scales [rows, cols/16], s_t as numpy float32)."""
    x_bits = np.asarray(x_bits, dtype=np.uint16)
    rows, cols = x_bits.shape
    vals = [[bf16_exact(int(b)) for b in row] for row in x_bits]
    amax_t = max(abs(v) for row in vals for v in row)
    s_t = rn_binary32(amax_t / 2688)
    t = rn_binary32(6 * s_t)
    codes = np.zeros((rows, cols // 2), dtype=np.uint8)
    scales = np.zeros((rows, cols // 16), dtype=np.uint8)
    key = [seed & M32, (seed >> 32) & M32] if seed is not None else None
    for r in range(rows):
        for j in range(cols // 16):
            blk = vals[r][16 * j:16 * j + 16]
            sb = 0 if s_t == 0 else e4m3_rne_satfinite(rn_binary32(max(abs(v) for v in blk) / t))
            scales[r, j] = sb
            if sb == 0:
                continue                      # codes 0x0
            den = rn_binary32(E4M3_GRID[sb] * s_t)
            draw = philox4x32([j, r, direction, 0], key, rounds) if key is not None else None
            for i, v in enumerate(blk):
                q = rn_binary32(v / den)
                neg = bool(x_bits[r, 16 * j + i] >> 15)
                if draw is None:
                    c = e2m1_rne(abs(q), neg)
                else:
                    c = e2m1_sr(abs(q), neg, (draw[i // 4] >> (8 * (i % 4))) & 0xFF)
                col = 16 * j + i
                codes[r, col // 2] |= c << (4 * (col % 2))
    return codes, scales, np.float32(float(s_t))


# ----------------------------------------------------------------- inputs

def _bf16_of(values) -> np.ndarray:
    return synth.f32_to_bf16_bits(np.asarray(values, dtype=np.float32))


def _random_tensor(seed):
    """N(0,1) rows with per-block magnitudes spread over 2^-12..2^6 (block scales
    across the E4M3 range, subnormal ones included), some zero blocks, -0.0
    entries; tensor max not a power of two."""
    rng = np.random.default_rng(seed)
    x = synth.bf16_bits_to_f32(synth.bf16_normal(16, 256, 1.0, seed=seed)).astype(np.float64)
    x = x.reshape(16, 16, 16) * np.exp2(rng.integers(-12, 7, size=(16, 16, 1)))
    x[3, 5] = 0.0
    x[7, 2] = -0.0
    x[0, 0, 0] = 93.5                      # tensor max; 93.5 / 2688 is not a power of two
    return _bf16_of(x.reshape(16, 256))


def _ulp32(v: float) -> float:
    return float(np.spacing(np.float32(abs(v))))


def _e2m1_adversarial(count, seed):
    """Tensors [1, 32]: block 0 holds the tensor max a alone; block 1 holds its
    max amax_b and a value x whose binary32 quotient x / den lies within one ulp
    of an E2M1 rounding midpoint (found by a vectorised binary32 search; the
    expected bytes come from the exact restatement, not from this search)."""
    rng = np.random.default_rng(seed)
    n = 1 << 20
    a = synth.bf16_bits_to_f32(rng.integers(0x3C00, 0x4300, n).astype(np.uint16))   # 2^-7..128
    amax_b = a * rng.uniform(0.01, 1.0, n).astype(np.float32)
    amax_b = synth.bf16_bits_to_f32(_bf16_of(amax_b))
    s_t = a / np.float32(2688)
    not_pow2 = np.frexp(s_t)[0] != 0.5
    t = np.float32(6) * s_t
    ratio = amax_b / t
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0], np.float32)
    grid = np.array([float(g) for g in E4M3_GRID], np.float64)
    sb = np.abs(ratio.astype(np.float64)[:, None] - grid[None, 1:]).argmin(axis=1) + 1
    den = grid[sb].astype(np.float32) * s_t
    out = []
    for mid in mids:
        # BF16 x nearest mid * den; keep three kinds of quotient near the midpoint:
        # rounded onto it from off it, one ulp beside it, and exactly on it
        x = synth.bf16_bits_to_f32(_bf16_of(mid * den))
        q = x / den
        exact = x.astype(np.float64) / den.astype(np.float64)
        ok = (np.abs(q - mid) <= np.spacing(mid)) & (x <= amax_b) & (x > 0) & not_pow2
        kinds = [ok & (q == mid) & (exact != mid), ok & (q != mid), ok & (exact == mid)]
        for kind in kinds:
            for i in np.flatnonzero(kind)[:2]:
                out.append((a[i], amax_b[i], x[i]))
    rng.shuffle(out)
    tensors = []
    for a_i, b_i, x_i in out[:count]:
        blk1 = [b_i, x_i, -x_i] + [x_i * 0.5] * 13
        tensors.append(_bf16_of([[a_i] + [0.0] * 15 + blk1]))
    return tensors


def _e4m3_adversarial(count, seed):
    """Tensors [1, 32] whose block-1 ratio amax_b / t lies within one binary32 ulp
    of a midpoint of two neighbouring E4M3 values."""
    rng = np.random.default_rng(seed)
    n = 1 << 20
    a = synth.bf16_bits_to_f32(rng.integers(0x3C00, 0x4300, n).astype(np.uint16))
    s_t = a / np.float32(2688)
    not_pow2 = np.frexp(s_t)[0] != 0.5
    t = np.float32(6) * s_t
    grid = np.array([float(g) for g in E4M3_GRID], np.float64)
    mid_all = ((grid[1:] + grid[:-1]) / 2).astype(np.float32)   # exact in binary32
    pick = rng.integers(0, len(mid_all), n)
    mid = mid_all[pick]
    out = []
    for step in (-1, 0, 1):
        bb = _bf16_of(mid * t).astype(np.int64) + step
        b = synth.bf16_bits_to_f32(bb.astype(np.uint16))
        r = b / t
        hit = (np.abs(r - mid) <= np.spacing(mid)) & (b <= a) & (b > 0) & not_pow2
        for i in np.flatnonzero(hit)[:count]:
            out.append((a[i], b[i]))
    rng.shuffle(out)
    tensors = []
    for a_i, b_i in out[:count]:
        blk1 = [b_i] + list(np.linspace(-b_i, b_i, 15, dtype=np.float32))
        tensors.append(_bf16_of([[a_i] + [0.0] * 15 + blk1]))
    return tensors


def _exact_ties():
    """Quotients exactly on E2M1 midpoints under a non-power-of-two s_t: the tensor
    max 63 gives s_t = 63 / 2688 = 3 / 128 exactly, so den = E4M3(sb) * 3 / 128
    is exact, 1 / den is not, and x = mid * den is a BF16 value."""
    out = []
    for amax_b in (7.0, 10.5, 40.0, 63.0):
        s_t = Fraction(3, 128)
        sb = e4m3_rne_satfinite(rn_binary32(Fraction(amax_b) / rn_binary32(6 * s_t)))
        den = E4M3_GRID[sb] * s_t
        xs = [float(m * den) for m in (Fraction(1, 4), Fraction(3, 4), Fraction(5, 4),
                                       Fraction(7, 4), Fraction(5, 2), Fraction(7, 2),
                                       Fraction(5))]
        xs = [v for v in xs if v <= amax_b][:15]
        blk1 = [amax_b] + xs + [-v for v in xs]
        blk1 = (blk1 + [0.0] * 16)[:16]
        x = _bf16_of([[63.0] + [0.0] * 15 + blk1])
        assert all(float(bf16_exact(int(b))) == v for b, v in zip(x[0, 16:], blk1))
        out.append(x)
    return out


def _cases():
    cases = [("random", t) for t in (_random_tensor(31), _random_tensor(32))]
    cases += [("normal", synth.bf16_normal(8, 512, 1.0, seed=33))]
    cases += [("e2m1-midpoint", t) for t in _e2m1_adversarial(42, seed=34)]
    cases += [("e4m3-midpoint", t) for t in _e4m3_adversarial(24, seed=35)]
    cases += [("exact-tie", t) for t in _exact_ties()]
    return cases


CASES = _cases()


def test_adversarial_sets_are_not_empty():
    kinds = [k for k, _ in CASES]
    assert kinds.count("e2m1-midpoint") >= 30 and kinds.count("e4m3-midpoint") >= 20
    # s_t is not a power of two in any case
    for _, x in CASES:
        amax = max(abs(bf16_exact(int(b))) for b in x.ravel())
        s_t = rn_binary32(amax / 2688)
        assert s_t.numerator & (s_t.numerator - 1) != 0 or s_t.denominator & (s_t.denominator - 1) != 0


def test_rn_binary32_agrees_with_ieee_division_on_samples():
    """A check of the restatement's rounding itself: on random binary32 operands,
    RN of the exact quotient equals numpy's IEEE binary32 division."""
    rng = np.random.default_rng(5)
    a = rng.standard_normal(2000).astype(np.float32)
    b = (rng.standard_normal(2000) * 7).astype(np.float32)
    for x, y in zip(a, b):
        assert rn_binary32(Fraction(float(x)) / Fraction(float(y))) == Fraction(float(x / y))


def test_oracle_nvfp4_matches_exact_restatement(oracle):
    for kind, x in CASES:
        codes, scales, s_t = oracle.nvfp4_quantize(x)
        e_codes, e_scales, e_st = nvfp4_exact(x)
        assert s_t.tobytes() == e_st.tobytes(), kind
        assert np.array_equal(scales, e_scales), kind
        assert np.array_equal(codes, e_codes), kind


@pytest.mark.parametrize("seed,rounds,direction", [(0x5EED, 10, 0), (0x1234567890AB, 7, 1)])
def test_oracle_nvfp4_sr_matches_exact_restatement(oracle, seed, rounds, direction):
    for kind, x in CASES:
        codes, scales, s_t = oracle.nvfp4_quantize_sr(x, seed, rounds, direction)
        e_codes, e_scales, e_st = nvfp4_exact(x, seed=seed, rounds=rounds, direction=direction)
        assert s_t.tobytes() == e_st.tobytes(), kind
        assert np.array_equal(scales, e_scales), kind
        assert np.array_equal(codes, e_codes), kind
