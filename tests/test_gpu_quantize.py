"""GPU parity of the quantize pre-pass and the scale re-layout: byte-equal to
the CPU oracle (codes, scales, NVFP4 tensor scale)."""
import numpy as np
import pytest

import block_scaled_fp4_bf16_gb300 as mx
import oracle
from block_scaled_fp4_bf16_gb300 import synth
from tests.gpu_helpers import (gpu_quantize, gpu_quantize_2d, gpu_quantize_group, gpu_quantize_nv2d,
                               gpu_quantize_sr, gpu_relayout)

pytestmark = pytest.mark.gpu

MX, NV = mx.MX_FMT_MXFP4, mx.MX_FMT_NVFP4
PLAIN, TILED = mx.MX_SCALE_PLAIN, mx.MX_SCALE_TCGEN05


def _unpack(c):
    c = np.asarray(c, np.uint8)
    out = np.empty(c.shape[:-1] + (c.shape[-1] * 2,), np.uint8)
    out[..., 0::2] = c & 0xF
    out[..., 1::2] = c >> 4
    return out


def _explain(x, codes, ref_codes, scales, ref_scales, blk):
    """Assertion text naming the first mismatching elements and their blocks."""
    g, r = _unpack(codes), _unpack(ref_codes)
    bad = np.argwhere(g != r)
    lines = [f"{len(bad)} code mismatches"]
    xf = synth.bf16_bits_to_f32(x)
    for row, col in bad[:6]:
        j = col // blk
        lines.append(f"  [{row},{col}] x={xf[row, col]!r} gpu={g[row, col]} oracle={r[row, col]} "
                     f"block_amax={np.abs(xf[row, j * blk:(j + 1) * blk]).max()!r}")
    return "\n".join(lines)


def _check_mx(x, layout=PLAIN, ld=None):
    codes, scales, _ = gpu_quantize(x, MX, layout, ld=ld)
    rc, rs = oracle.mx_quantize(x)
    assert np.array_equal(codes, rc), _explain(x, codes, rc, scales, rs, 32)
    if layout == PLAIN:
        assert np.array_equal(scales.reshape(rs.shape), rs)
    else:
        assert np.array_equal(scales, oracle.scale_tile(rs))


def _check_nv(x, layout=PLAIN, ld=None):
    codes, scales, s_t = gpu_quantize(x, NV, layout, ld=ld)
    rc, rs, rt = oracle.nvfp4_quantize(x)
    assert np.float32(s_t).view(np.uint32) == np.float32(rt).view(np.uint32)
    if layout == PLAIN:
        bad_s = np.argwhere(scales.reshape(rs.shape) != rs)
    else:
        bad_s = np.argwhere(scales != oracle.scale_tile(rs))
    assert np.array_equal(codes, rc), (f"scale mismatches {len(bad_s)} first {bad_s[:4].tolist()}; "
                                       + _explain(x, codes, rc, scales, rs, 16)
                                       + f"\n  s_t={float(rt)!r}")
    assert len(bad_s) == 0


@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 96), (33, 160), (128, 256), (129, 4096),
                                       (200, 64), (517, 1024)])
@pytest.mark.parametrize("layout", [PLAIN, TILED])
def test_mx_quantize_ragged_shapes(rows, cols, layout):
    x = synth.bf16_normal(rows, cols, 1.0, seed=rows * 131 + cols)
    _check_mx(x, layout)


def test_mx_quantize_leading_dim():
    x = synth.bf16_normal(70, 256, 3.0, seed=5)
    _check_mx(x, PLAIN, ld=264)
    _check_mx(x, TILED, ld=512)


def test_mx_quantize_exhaustive_bf16():
    """Every finite BF16 value, as its block's max and under a larger anchor."""
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = b[((b >> 7) & 0xFF) != 0xFF]
    x = np.zeros((v.size, 64), np.uint16)
    x[:, 0] = v
    x[:, 33] = v
    x[:, 40] = synth.f32_to_bf16_bits(np.array([1.75 * 2.0 ** 9], np.float32))[0]
    x[:, 5] = v ^ 0x8000
    _check_mx(x, PLAIN)
    _check_mx(x, TILED)


def test_mx_quantize_special_blocks():
    x = synth.bf16_normal(64, 512, 1.0, seed=9)
    x[0, :32] = 0
    x[1, 32:64] = 0x8000               # -0 block
    x[2, :] = synth.f32_to_bf16_bits(np.full(512, 1e-40, np.float32))  # subnormals
    x[3, :32] = 0x7F7F                 # largest finite
    x[4, 64:96] = 0x0001               # smallest subnormal
    x[5, ::7] = synth.f32_to_bf16_bits(np.array([5.0 * 2 ** -20], np.float32))[0]
    _check_mx(x, PLAIN)
    _check_mx(x, TILED)


def test_mx_quantize_llm_shapes_full_size():
    """The quantize+GEMM and MLP up-projection operands at their full sizes."""
    for name in ["quant_gemm_2048x4096x4096", "mlp_up_16384x28672x8192"]:
        w = synth.workload_inputs(name)
        _check_mx(w["a"], TILED)
        _check_mx(w["b"], TILED)
        del w


@pytest.mark.parametrize("rows,cols", [(1, 16), (5, 48), (128, 256), (300, 1024)])
@pytest.mark.parametrize("layout", [PLAIN, TILED])
def test_nvfp4_quantize_ragged_shapes(rows, cols, layout):
    x = synth.bf16_normal(rows, cols, 1.0, seed=rows * 17 + cols)
    _check_nv(x, layout)


def test_nvfp4_quantize_full_size():
    w = synth.workload_inputs("nvfp4_4096x4096x4096")
    _check_nv(w["a"], TILED)
    _check_nv(w["b"], TILED)


def test_nvfp4_quantize_special_cases():
    x = synth.bf16_normal(40, 256, 2.0, seed=3)
    x[0, :16] = 0
    x[1, 16:32] = 0x8000
    x[2, :] = synth.f32_to_bf16_bits(np.full(256, 1e-30, np.float32))  # blocks whose sb rounds to 0
    x[3, 0] = synth.f32_to_bf16_bits(np.array([1000.0], np.float32))[0]
    _check_nv(x, PLAIN)
    _check_nv(np.zeros((4, 64), np.uint16), PLAIN)      # all zero: s_t = 0
    # exhaustive BF16 values against a fixed tensor max
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = b[(((b >> 7) & 0xFF) != 0xFF) & ((b & 0x7FFF) < 0x4700)]
    y = np.zeros((v.size, 16), np.uint16)
    y[:, 3] = v
    y[:, 9] = 0x4000
    y[0, 0] = 0x4700
    _check_nv(y, PLAIN)


@pytest.mark.parametrize("rows,cols,fmt", [(128, 256, MX), (33, 96, MX), (300, 1024, MX),
                                           (64, 64, NV), (257, 512, NV)])
def test_scale_relayout_matches_oracle(rows, cols, fmt):
    blk = 32 if fmt == MX else 16
    plain = np.random.default_rng(rows + cols).integers(0, 256, size=(rows, cols // blk),
                                                        dtype=np.uint8)
    tiled = gpu_relayout(plain, rows, cols, fmt).cpu().numpy()
    assert np.array_equal(tiled, oracle.scale_tile(plain))


def _finite_bf16_upto(limit: float) -> np.ndarray:
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = ((b >> 7) & 0xFF) != 0xFF
    vals = synth.bf16_bits_to_f32(b)
    return b[finite & (np.abs(vals) <= limit)]


@pytest.mark.parametrize("tmax", [1.0, 3.0, 448.0, 1000.0, 1.5e-3, 7.5e5, 3e30, 2e-30])
def test_nvfp4_quantize_every_bf16_under_many_divisors(tmax):
    """Each finite BF16 value v (|v| <= block max) quantized in blocks whose
    divisor E4M3(sb) * s_t takes many values: the per-block correctly rounded
    division must agree byte for byte with the oracle's binary32 division."""
    rows = []
    for k in (0, 1, 3, 6, 9, 13):
        for mant in (1.0, 1.375, 1.875):
            bmax = tmax * 2.0 ** -k * mant / 1.875
            bb = synth.f32_to_bf16_bits(np.array([bmax], np.float32))[0]
            bval = float(synth.bf16_bits_to_f32(np.array([bb], np.uint16))[0])
            v = _finite_bf16_upto(bval)
            y = np.zeros((v.size, 16), np.uint16)
            y[:, 0] = bb
            y[:, 7] = v
            rows.append(y)
    x = np.concatenate(rows)
    x[0, 15] = synth.f32_to_bf16_bits(np.array([tmax], np.float32))[0]
    _check_nv(x, PLAIN)


def test_leading_dim_not_32_byte_aligned():
    """ld % 16 != 0 takes the 16-byte load path (x is only 16-byte aligned per row)."""
    x = synth.bf16_normal(96, 512, 1.0, seed=31)
    _check_mx(x, TILED, ld=520)
    _check_nv(x, TILED, ld=520)
    _check_nv(x, PLAIN, ld=528)


# ---- grouped quantize: one launch, each tensor byte-equal to the oracle ----

def _group_inputs(shapes, seed):
    return [synth.bf16_normal(r, c, 0.5 + i, seed=seed + i) for i, (r, c) in enumerate(shapes)]


@pytest.mark.parametrize("layout", [PLAIN, TILED])
def test_mx_quantize_group_matches_oracle(layout):
    shapes = [(129, 4096), (3, 96), (256, 512), (1, 32), (517, 1024)]
    xs = _group_inputs(shapes, 700)
    xs[2][5, :32] = 0                      # a zero block inside the group
    got = gpu_quantize_group(xs, MX, layout, lds=[None, 104, None, 40, 1032])
    for x, (codes, scales, s_t) in zip(xs, got):
        rc, rs = oracle.mx_quantize(x)
        assert s_t is None
        assert np.array_equal(codes, rc), _explain(x, codes, rc, scales, rs, 32)
        want = rs.ravel() if layout == PLAIN else oracle.scale_tile(rs)
        assert np.array_equal(scales, want)


@pytest.mark.parametrize("layout", [PLAIN, TILED])
def test_nvfp4_quantize_group_matches_oracle(layout):
    """Each tensor gets its own amax and s_t although the group shares launches."""
    shapes = [(300, 1024), (5, 48), (128, 256)]
    xs = _group_inputs(shapes, 800)
    xs[1] = xs[1] * 0                     # an all-zero tensor: s_t = 0, codes 0
    xs[2][7, 3] = synth.f32_to_bf16_bits(np.array([1000.0], np.float32))[0]
    got = gpu_quantize_group(xs, NV, layout)
    for x, (codes, scales, s_t) in zip(xs, got):
        rc, rs, rt = oracle.nvfp4_quantize(x)
        assert np.float32(s_t).view(np.uint32) == np.float32(rt).view(np.uint32)
        assert np.array_equal(codes, rc), _explain(x, codes, rc, scales, rs, 16)
        want = rs.ravel() if layout == PLAIN else oracle.scale_tile(rs)
        assert np.array_equal(scales, want)


def test_quantize_group_of_the_largest_size_matches_single_calls():
    n = mx.MX_QUANTIZE_GROUP_MAX
    xs = _group_inputs([(64 + 32 * i, 256 + 128 * i) for i in range(n)], 900)
    for fmt in (MX, NV):
        got = gpu_quantize_group(xs, fmt, TILED)
        for x, (codes, scales, s_t) in zip(xs, got):
            c1, s1, t1 = gpu_quantize(x, fmt, TILED)
            assert np.array_equal(codes, c1) and np.array_equal(scales, s1)
            assert (s_t is None and t1 is None) or s_t.view(np.uint32) == t1.view(np.uint32)


def test_quantize_group_at_the_quantize_gemm_workload_size():
    """The activation 2048x4096 and weight 4096x4096 of the quantize+GEMM
    workload in one call, as the benchmark issues them."""
    w = synth.workload_inputs("quant_gemm_2048x4096x4096")
    got = gpu_quantize_group([w["a"], w["b"]], MX, TILED)
    for x, (codes, scales, _) in zip([w["a"], w["b"]], got):
        rc, rs = oracle.mx_quantize(x)
        assert np.array_equal(codes, rc)
        assert np.array_equal(scales, oracle.scale_tile(rs))


# ---- bidimensional quantize: rowwise and columnwise outputs byte-equal ------

def _check_2d(x, layout, ld=None):
    codes, scales, codes_t, scales_t = gpu_quantize_2d(x, layout, ld=ld)
    rc, rs, rct, rst = oracle.mx_quantize_2d(x)
    assert np.array_equal(codes, rc), "rowwise codes: " + _explain(x, codes, rc, scales, rs, 32)
    assert np.array_equal(codes_t, rct), "columnwise codes: " + _explain(
        np.ascontiguousarray(x.T), codes_t, rct, scales_t, rst, 32)
    if layout == PLAIN:
        assert np.array_equal(scales, rs.ravel()) and np.array_equal(scales_t, rst.ravel())
    else:
        assert np.array_equal(scales, oracle.scale_tile(rs))
        assert np.array_equal(scales_t, oracle.scale_tile(rst))


@pytest.mark.parametrize("rows,cols", [(32, 32), (64, 96), (96, 256), (128, 512), (160, 288),
                                       (544, 1024), (256, 4096), (4096, 288)])
@pytest.mark.parametrize("layout", [PLAIN, TILED])
def test_mx_quantize_2d_matches_oracle(rows, cols, layout):
    x = synth.bf16_normal(rows, cols, 1.0, seed=rows * 7 + cols)
    x[0, :32] = 0                                     # zero row block
    x[:32, min(5, cols - 1)] = 0x8000                 # column block of -0
    _check_2d(x, layout)


def test_mx_quantize_2d_leading_dim_and_special_values():
    x = synth.bf16_normal(96, 160, 3.0, seed=41)
    x[2, :] = synth.f32_to_bf16_bits(np.full(160, 1e-40, np.float32))   # subnormals
    x[:, 3] = 0x7F7F                                                   # largest finite
    x[40:64, 70] = 0x0001
    _check_2d(x, TILED, ld=168)                      # 16-byte (not 32-byte) aligned rows
    _check_2d(x, PLAIN, ld=256)


def test_mx_quantize_2d_full_size_weight():
    """The 4096 x 4096 weight of the quantize+GEMM workload."""
    w = synth.workload_inputs("quant_gemm_2048x4096x4096")
    _check_2d(w["b"], TILED)


def test_mx_quantize_2d_columnwise_only():
    """Rowwise outputs omitted (null): the columnwise output is unchanged."""
    x = synth.bf16_normal(192, 320, 1.0, seed=43)
    _, _, rct, rst = oracle.mx_quantize_2d(x)
    for layout in (PLAIN, TILED):
        codes, scales, codes_t, scales_t = gpu_quantize_2d(x, layout, columnwise_only=True)
        assert codes is None and scales is None
        assert np.array_equal(codes_t, rct)
        assert np.array_equal(scales_t, rst.ravel() if layout == PLAIN else oracle.scale_tile(rst))


# ---------------------------------------------------------------- stochastic rounding (NVFP4)

def _check_nv_sr(x, seed, rounds=10, layout=PLAIN, ld=None):
    codes, scales, s_t = gpu_quantize_sr(x, seed, rounds, layout, ld)
    rc, rs, rt = oracle.nvfp4_quantize_sr(x, seed, rounds)
    assert np.float32(s_t).view(np.uint32) == np.float32(rt).view(np.uint32)
    if layout == PLAIN:
        assert np.array_equal(scales.reshape(rs.shape), rs)
    else:
        assert np.array_equal(scales, oracle.scale_tile(rs))
    assert np.array_equal(codes, rc), _explain(x, codes, rc, scales, rs, 16) + f"\n  seed={seed}"
    return codes


@pytest.mark.parametrize("rows,cols", [(1, 16), (5, 48), (128, 256), (300, 1024), (129, 4096)])
@pytest.mark.parametrize("layout", [PLAIN, TILED])
def test_nvfp4_sr_matches_oracle(rows, cols, layout):
    x = synth.bf16_normal(rows, cols, 1.0, seed=rows * 31 + cols)
    _check_nv_sr(x, 0x5EED0000 + rows, 10, layout)


@pytest.mark.parametrize("seed", [0, 1, 0xFFFFFFFF, 0x100000000, 0xFEDCBA9876543210])
@pytest.mark.parametrize("rounds", [1, 2, 7, 10, 16])
def test_nvfp4_sr_seeds_and_round_counts(seed, rounds):
    x = synth.bf16_normal(64, 512, 0.02, seed=7)
    _check_nv_sr(x, seed, rounds)


def test_nvfp4_sr_full_size():
    w = synth.workload_inputs("nvfp4_4096x4096x4096")
    _check_nv_sr(w["a"], 42, 10, TILED)
    _check_nv_sr(w["b"], 43, 10, TILED)


def test_nvfp4_sr_special_cases_and_unaligned_rows():
    x = synth.bf16_normal(40, 256, 2.0, seed=3)
    x[0, :16] = 0
    x[1, 16:32] = 0x8000
    x[2, :] = synth.f32_to_bf16_bits(np.full(256, 1e-30, np.float32))
    x[3, 0] = synth.f32_to_bf16_bits(np.array([1000.0], np.float32))[0]
    _check_nv_sr(x, 11)
    _check_nv_sr(x, 12, ld=264)          # rows only 16-byte aligned: the two-load path
    _check_nv_sr(np.zeros((4, 64), np.uint16), 13)


@pytest.mark.parametrize("tmax", [1.0, 448.0, 1.5e-3, 7.5e5, 3e30, 2e-30])
def test_nvfp4_sr_every_bf16_under_many_divisors(tmax):
    """Every finite BF16 value under many block divisors (including divisors
    outside the reciprocal's safe range, which take the IEEE division)."""
    rows = []
    for k in (0, 1, 3, 6, 9, 13):
        for mant in (1.0, 1.375, 1.875):
            bmax = tmax * 2.0 ** -k * mant / 1.875
            bb = synth.f32_to_bf16_bits(np.array([bmax], np.float32))[0]
            bval = float(synth.bf16_bits_to_f32(np.array([bb], np.uint16))[0])
            v = _finite_bf16_upto(bval)
            y = np.zeros((v.size, 16), np.uint16)
            y[:, 0] = bb
            y[:, 7] = v
            y[:, 12] = v[::-1]
            rows.append(y)
    x = np.concatenate(rows)
    x[0, 15] = synth.f32_to_bf16_bits(np.array([tmax], np.float32))[0]
    _check_nv_sr(x, int(tmax * 1000) & 0xFFFF)


def test_nvfp4_sr_is_deterministic_and_unbiased_on_the_gpu():
    """Same seed, same bytes; the mean over 128 seeds of the dequantized codes
    is within 5 standard errors (plus the 1/256-step bias) of x / den."""
    x = synth.bf16_normal(32, 256, 0.5, seed=21)
    a = gpu_quantize_sr(x, 99)[0]
    assert np.array_equal(a, gpu_quantize_sr(x, 99)[0])
    assert not np.array_equal(a, gpu_quantize_sr(x, 100)[0])
    _, rs, rt = oracle.nvfp4_quantize(x)
    e4 = np.array([oracle.e4m3_decode(b) for b in range(256)])
    den = np.repeat((e4[rs] * np.float64(rt)).astype(np.float32), 16, axis=1)
    q = (synth.bf16_bits_to_f32(x) / den).astype(np.float64)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6])
    n, acc = 128, np.zeros_like(q)
    for seed in range(n):
        c = _unpack(gpu_quantize_sr(x, 5000 + seed)[0])
        acc += np.where(c & 8, -1.0, 1.0) * grid[c & 7]
    step = np.where(np.abs(q) < 2, 0.5, np.where(np.abs(q) < 4, 1.0, 2.0))
    assert np.all(np.abs(acc / n - q) <= step * (5 * 0.5 / np.sqrt(n) + 1 / 256))


# ---------------------------------------------------------------- bidimensional NVFP4

def _check_nv2d(x, layout, ld=None, seed=None, rounds=10):
    codes, scales, codes_t, scales_t, s_t = gpu_quantize_nv2d(x, layout, ld=ld, seed=seed,
                                                             rounds=rounds)
    rc, rs, rct, rst, rt = oracle.nvfp4_quantize_2d(x, seed=seed, rounds=rounds)
    assert np.float32(s_t).view(np.uint32) == np.float32(rt).view(np.uint32)
    assert np.array_equal(codes, rc), "rowwise codes: " + _explain(x, codes, rc, scales, rs, 16)
    assert np.array_equal(codes_t, rct), "columnwise codes: " + _explain(
        np.ascontiguousarray(x.T), codes_t, rct, scales_t, rst, 16)
    if layout == PLAIN:
        assert np.array_equal(scales, rs.ravel()) and np.array_equal(scales_t, rst.ravel())
    else:
        assert np.array_equal(scales, oracle.scale_tile(rs))
        assert np.array_equal(scales_t, oracle.scale_tile(rst))


@pytest.mark.parametrize("rows,cols", [(16, 16), (32, 48), (64, 96), (96, 256), (160, 288),
                                       (544, 1040), (256, 4096), (4096, 272)])
@pytest.mark.parametrize("layout", [PLAIN, TILED])
@pytest.mark.parametrize("seed", [None, 0x5EED])
def test_nvfp4_quantize_2d_matches_oracle(rows, cols, layout, seed):
    x = synth.bf16_normal(rows, cols, 1.0, seed=rows * 5 + cols)
    x[0, :16] = 0                                     # zero row block
    x[:16, min(5, cols - 1)] = 0x8000                 # column block of -0
    _check_nv2d(x, layout, seed=seed)


def test_nvfp4_quantize_2d_leading_dim_special_values_and_rounds():
    x = synth.bf16_normal(96, 160, 3.0, seed=51)
    x[2, :] = synth.f32_to_bf16_bits(np.full(160, 1e-40, np.float32))   # subnormals
    x[:, 3] = 0x7F7F                                                   # largest finite
    x[40:64, 70] = 0x0001
    _check_nv2d(x, TILED, ld=168)                    # 16-byte (not 32-byte) aligned rows
    _check_nv2d(x, PLAIN, ld=256, seed=7)
    _check_nv2d(x, TILED, seed=0xFFFFFFFF00000001, rounds=7)
    _check_nv2d(np.zeros((32, 64), np.uint16), PLAIN, seed=3)          # s_t = 0


def test_nvfp4_quantize_2d_rowwise_equals_one_dimensional_calls():
    """The rowwise output equals mx_quantize_bf16 / nvfp4_quantize_bf16_sr on x,
    the columnwise output equals them on x^T with direction 1 (oracle) and the
    same s_t."""
    x = synth.bf16_normal(128, 192, 0.5, seed=52)
    c, s, ct, st, ts = gpu_quantize_nv2d(x, TILED)
    c1, s1, t1 = gpu_quantize(x, NV, TILED)
    ct1, st1, tt1 = gpu_quantize(np.ascontiguousarray(x.T), NV, TILED)
    assert np.array_equal(c, c1) and np.array_equal(s, s1) and ts == t1
    assert np.array_equal(ct, ct1) and np.array_equal(st, st1) and tt1 == ts
    c, s, ct, st, ts = gpu_quantize_nv2d(x, PLAIN, seed=99)
    c1, s1, t1 = gpu_quantize_sr(x, 99, 10, PLAIN)
    assert np.array_equal(c, c1) and np.array_equal(s, s1) and ts == t1


def test_nvfp4_quantize_2d_full_size():
    """The 16384 x 8192 tensor of the stochastic-rounding workload, both roundings."""
    x = synth.workload_inputs("nvfp4_sr_16384x8192")["a"]
    _check_nv2d(x, TILED, seed=0x5EED5EED)
    _check_nv2d(x, TILED)


def test_nvfp4_quantize_2d_more_tiles_than_resident_ctas():
    """With stochastic rounding the kernel is persistent (4 CTAs per SM, each
    taking every grid-th 64 x 256 tile): 701 tiles of a narrow tensor, the last
    one ragged (16 of its 64 rows), so that some CTAs take two tiles."""
    x = synth.bf16_normal(64 * 700 + 16, 32, 1.0, seed=54)
    x[-16:, :16] = 0                                  # a zero block in the ragged tile
    for layout in (PLAIN, TILED):
        _check_nv2d(x, layout, seed=0x5EED)
    _check_nv2d(x, TILED)


def test_nvfp4_quantize_2d_columnwise_only():
    x = synth.bf16_normal(192, 320, 1.0, seed=53)
    for seed in (None, 17):
        _, _, rct, rst, rt = oracle.nvfp4_quantize_2d(x, seed=seed)
        for layout in (PLAIN, TILED):
            codes, scales, codes_t, scales_t, ts = gpu_quantize_nv2d(x, layout, columnwise_only=True,
                                                                    seed=seed)
            assert codes is None and scales is None and ts == rt
            assert np.array_equal(codes_t, rct)
            assert np.array_equal(scales_t, rst.ravel() if layout == PLAIN else oracle.scale_tile(rst))


def test_nvfp4_sr_full_size_bench_tensor():
    """The 16384 x 8192 tensor of the stochastic-rounding workload, in the tile
    scale order and with the seed bench.py uses."""
    x = synth.workload_inputs("nvfp4_sr_16384x8192")["a"]
    _check_nv_sr(x, 0x5EED5EED, 10, TILED)
