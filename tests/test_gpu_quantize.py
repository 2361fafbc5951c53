"""GPU parity of the quantize pre-pass and the scale re-layout: byte-equal to
the CPU oracle (codes, scales, NVFP4 tensor scale)."""
import numpy as np
import pytest

import block_scaled_fp4_bf16_gb300 as mx
import oracle
from block_scaled_fp4_bf16_gb300 import synth
from tests.gpu_helpers import gpu_quantize, gpu_relayout

pytestmark = pytest.mark.gpu

MX, NV = mx.MX_FMT_MXFP4, mx.MX_FMT_NVFP4
PLAIN, TILED = mx.MX_SCALE_PLAIN, mx.MX_SCALE_TCGEN05


def _check_mx(x, layout=PLAIN, ld=None):
    codes, scales, _ = gpu_quantize(x, MX, layout, ld=ld)
    rc, rs = oracle.mx_quantize(x)
    assert np.array_equal(codes, rc)
    if layout == PLAIN:
        assert np.array_equal(scales.reshape(rs.shape), rs)
    else:
        assert np.array_equal(scales, oracle.scale_tile(rs))


def _check_nv(x, layout=PLAIN, ld=None):
    codes, scales, s_t = gpu_quantize(x, NV, layout, ld=ld)
    rc, rs, rt = oracle.nvfp4_quantize(x)
    assert np.float32(s_t).view(np.uint32) == np.float32(rt).view(np.uint32)
    assert np.array_equal(codes, rc)
    if layout == PLAIN:
        assert np.array_equal(scales.reshape(rs.shape), rs)
    else:
        assert np.array_equal(scales, oracle.scale_tile(rs))


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
