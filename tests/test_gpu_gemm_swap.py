"""GPU parity of the swapped-operand GEMM kernel (M <= 64 with the automatic
split: D^T = B A^T on the tensor cores, K split over the CTAs of a cluster whose
partial sums meet in shared memory) against the CPU oracle, element by
element.  Shapes cover one 128-row weight block with most rows past N, ragged
N, many blocks, all three cluster sizes (1, 2, 4), both formats and both output
types; the result is bit-identical across runs (fixed order of the partial
sums) and agrees with the workspace split-K path within the tolerances."""
import numpy as np
import pytest

import block_scaled_fp4_bf16_gb300 as mx
import oracle
from block_scaled_fp4_bf16_gb300 import synth
from tests.gpu_helpers import check_bf16, check_fp32, gpu_gemm, gpu_quantize

pytestmark = pytest.mark.gpu

MX, NV = mx.MX_FMT_MXFP4, mx.MX_FMT_NVFP4
TILED = mx.MX_SCALE_TCGEN05


def _mx_case(m, n, k, seed):
    return (synth.fp4_codes(m, k, seed), synth.scale_bytes(m, k // 32, 120, 134, seed + 1),
            synth.fp4_codes(n, k, seed + 2), synth.scale_bytes(n, k // 32, 120, 134, seed + 3))


def _check(d, ref, s_abs, out_fp32, what):
    if out_fp32:
        check_fp32(d, ref, s_abs, what)
        assert np.count_nonzero(d) == np.count_nonzero(ref)
    else:
        check_bf16(d, ref, s_abs, what)


# (m, n, k): cluster of 1 (one stage; one block with 96 rows past N), of 2, of 4,
# ragged N, M = 64, and more 128-row blocks than SMs (two CTAs per SM, also
# with a ragged last block and with more blocks than two per SM hold); M = 64
# in clusters of 4 (a ragged last 128-row slice); 32-row slices in clusters of
# 4 and of 2 (the latter with a ragged last 128-row atom), and for M = 64 in
# clusters of 4 (one lane quarter of real output per CTA)
SHAPES = [(32, 32, 256), (32, 8192, 8192), (32, 4096, 4096), (64, 4224, 2048),
          (32, 1056, 1024), (64, 640, 1024), (32, 28672, 512), (64, 28672, 1024),
          (32, 24608, 2048), (32, 45056, 512), (64, 4096, 8192), (64, 2080, 8192),
          (32, 768, 4096), (64, 864, 2048), (64, 512, 8192)]


@pytest.mark.parametrize("m,n,k", SHAPES)
@pytest.mark.parametrize("out_fp32", [True, False])
def test_swap_mxfp4_matches_oracle(m, n, k, out_fp32):
    a, sa, b, sb = _mx_case(m, n, k, seed=m + n + k)
    d = gpu_gemm(MX, a, oracle.scale_tile(sa), b, oracle.scale_tile(sb), m, n, k, out_fp32)
    assert mx.mx_gemm_workspace_bytes(m, n, k, 0) == 0      # no scratch on this path
    ref, s_abs = oracle.mx_gemm(a, sa, b, sb, m, n, k)
    _check(d, ref, s_abs, out_fp32, f"swap mxfp4 {m}x{n}x{k}")


@pytest.mark.parametrize("m,n,k", [(32, 4096, 4096), (64, 1152, 2048), (32, 96, 512),
                                   (32, 28672, 1024), (64, 20480, 512), (64, 4096, 8192)])
@pytest.mark.parametrize("out_fp32", [True, False])
def test_swap_nvfp4_matches_oracle(m, n, k, out_fp32):
    xa = synth.bf16_normal(m, k, 1.0, seed=m * 3 + k)
    xb = synth.bf16_normal(n, k, 0.05, seed=n * 5 + k)
    ca, sa_t, ta = gpu_quantize(xa, NV, TILED)
    cb, sb_t, tb = gpu_quantize(xb, NV, TILED)
    ra, rsa, rta = oracle.nvfp4_quantize(xa)
    rb, rsb, rtb = oracle.nvfp4_quantize(xb)
    assert np.array_equal(ca, ra) and np.array_equal(cb, rb)
    d = gpu_gemm(NV, ca, sa_t, cb, sb_t, m, n, k, out_fp32, a_ts=ta, b_ts=tb)
    ref, s_abs = oracle.nvfp4_gemm(ra, rsa, rb, rsb, m, n, k, rta, rtb)
    _check(d, ref, s_abs, out_fp32, f"swap nvfp4 {m}x{n}x{k}")


@pytest.mark.parametrize("out_fp32", [True, False])
def test_swap_is_deterministic_and_agrees_with_the_workspace_path(out_fp32):
    m, n, k = 64, 4096, 8192            # a cluster of 4: three partials summed in order
    a, sa, b, sb = _mx_case(m, n, k, seed=91)
    ta, tb = oracle.scale_tile(sa), oracle.scale_tile(sb)
    d1 = gpu_gemm(MX, a, ta, b, tb, m, n, k, out_fp32)
    d2 = gpu_gemm(MX, a, ta, b, tb, m, n, k, out_fp32)
    assert np.array_equal(d1, d2)
    d_ws = gpu_gemm(MX, a, ta, b, tb, m, n, k, out_fp32, split_k=4)   # partials + reduce kernel
    ref, s_abs = oracle.mx_gemm(a, sa, b, sb, m, n, k)
    _check(d1, ref, s_abs, out_fp32, "swap, cluster of 4")
    _check(d_ws, ref, s_abs, out_fp32, "workspace split 4")


def test_swap_decode_mlp_workload_full_size():
    """The decode-shaped MLP up-projection (224 weight slices, two CTAs per SM)
    as the benchmark runs it, every output."""
    name = "decode_mlp_up_32x28672x8192"
    w = synth.workload_inputs(name)
    m, n, k = 32, 28672, 8192
    d = gpu_gemm(MX, w["a_codes"], oracle.scale_tile(w["a_scales"]), w["b_codes"],
                 oracle.scale_tile(w["b_scales"]), m, n, k, out_fp32=False)
    ref, s_abs = oracle.mx_gemm(w["a_codes"], w["a_scales"], w["b_codes"], w["b_scales"], m, n, k)
    stats = check_bf16(d, ref, s_abs, f"{name} (swapped kernel, two CTAs per SM)")
    assert stats["exact"] > 0.9 * stats["total"]


def test_swap_skinny_workload_full_size():
    """The decode-shaped workload as the benchmark runs it, every output."""
    w = synth.workload_inputs("skinny_32x8192x8192")
    m, n, k = 32, 8192, 8192
    d = gpu_gemm(MX, w["a_codes"], oracle.scale_tile(w["a_scales"]), w["b_codes"],
                 oracle.scale_tile(w["b_scales"]), m, n, k, out_fp32=False)
    ref, s_abs = oracle.mx_gemm(w["a_codes"], w["a_scales"], w["b_codes"], w["b_scales"], m, n, k)
    stats = check_bf16(d, ref, s_abs, "skinny 32x8192x8192 (swapped kernel)")
    assert stats["exact"] > 0.9 * stats["total"]


def test_swap_very_wide_weight():
    """N = 2^20 weight rows (8192 slices of 128, far more than two per SM hold),
    K = 256: the grid, the slice offsets and the output indices at a size where
    32-bit products of them would overflow; every output against the oracle."""
    m, n, k = 32, 1 << 20, 256
    a, sa, b, sb = _mx_case(m, n, k, seed=77)
    d = gpu_gemm(MX, a, oracle.scale_tile(sa), b, oracle.scale_tile(sb), m, n, k, out_fp32=False)
    ref, s_abs = oracle.mx_gemm(a, sa, b, sb, m, n, k)
    stats = check_bf16(d, ref, s_abs, "swap 32 x 2^20 x 256")
    assert stats["exact"] > 0.9 * stats["total"]
