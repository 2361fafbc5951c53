"""GPU parity of the block-scaled GEMM (MXFP4 and NVFP4) against the CPU oracle,
element by element at moderate sizes (several tiles, ragged tails) and on
sampled outputs at the full workload sizes, plus closed-form probes of the
scale and nibble conventions."""
import numpy as np
import pytest
import torch

import block_scaled_fp4_bf16_gb300 as mx
import oracle
from block_scaled_fp4_bf16_gb300 import synth
from tests.gpu_helpers import (bf16_bits_to_f64, check_bf16, check_fp32, check_guards, dev_u8,
                               gpu_gemm, gpu_quantize_2d, gpu_quantize, gpu_relayout, guarded,
                               sample_indices)

pytestmark = pytest.mark.gpu

MX, NV = mx.MX_FMT_MXFP4, mx.MX_FMT_NVFP4
TILED = mx.MX_SCALE_TCGEN05


def _codes_case(m, n, k, seed, lo=120, hi=134):
    return (synth.fp4_codes(m, k, seed), synth.scale_bytes(m, k // 32, lo, hi, seed + 1),
            synth.fp4_codes(n, k, seed + 2), synth.scale_bytes(n, k // 32, lo, hi, seed + 3))


def _run_and_check_mx(a, sa, b, sb, m, n, k, out_fp32, split_k=0):
    d = gpu_gemm(MX, a, oracle.scale_tile(sa), b, oracle.scale_tile(sb), m, n, k, out_fp32,
                 split_k=split_k)
    ref, s_abs = oracle.mx_gemm(a, sa, b, sb, m, n, k)
    what = f"mxfp4 {m}x{n}x{k} {'fp32' if out_fp32 else 'bf16'} split {split_k}"
    if out_fp32:
        check_fp32(d, ref, s_abs, what)
        assert np.count_nonzero(d) == np.count_nonzero(ref)
    else:
        check_bf16(d, ref, s_abs, what)
    return d


# ------------------------------------------------------------ closed forms

@pytest.mark.parametrize("m,n,k", [(128, 128, 256), (256, 512, 1024), (4096, 4096, 256)])
def test_all_ones_gives_k(m, n, k):
    a = np.full((m, k // 2), 0x22, np.uint8)          # code 2 = 1.0 in both nibbles
    b = np.full((n, k // 2), 0x22, np.uint8)
    s = lambda r: oracle.scale_tile(np.full((r, k // 32), 127, np.uint8))
    d = gpu_gemm(MX, a, s(m), b, s(n), m, n, k, out_fp32=True)
    assert np.all(d == k)


def test_scale_probe_rows_and_blocks():
    """A = B = 1.0 everywhere; D[m, n] = 32 * sum_j 2^(sa[m, j] - 127) * 2^(sb[n, j] - 127)."""
    m, n, k = 256, 256, 512
    rng = np.random.default_rng(1)
    sa = rng.integers(124, 131, size=(m, k // 32), dtype=np.uint8)
    sb = rng.integers(124, 131, size=(n, k // 32), dtype=np.uint8)
    ones = lambda r: np.full((r, k // 2), 0x22, np.uint8)
    d = gpu_gemm(MX, ones(m), oracle.scale_tile(sa), ones(n), oracle.scale_tile(sb), m, n, k,
                 out_fp32=True)
    ea = np.ldexp(1.0, sa.astype(np.int64) - 127)
    eb = np.ldexp(1.0, sb.astype(np.int64) - 127)
    assert np.array_equal(d.astype(np.float64), 32.0 * ea @ eb.T)


def test_k_position_probe():
    """Row r of A holds 1.0 at k = 2r and 2.0 at k = 2r + 1, nothing else; B is random.
    D[r, n] = B[n, 2r] + 2 B[n, 2r + 1] pins where each K element lands (the
    nibble order itself cancels in a dot product when A and B share it)."""
    m, n, k = 128, 128, 256
    a = np.zeros((m, k), np.uint8)
    a[np.arange(m), np.arange(m) * 2 % k] = 2       # even k in rows 0..127
    a[np.arange(m), (np.arange(m) * 2 + 1) % k] = 4  # and 2.0 at the odd k after it
    bcodes = np.random.default_rng(2).integers(0, 16, size=(n, k), dtype=np.uint8)
    pack = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8)
    s = lambda r: oracle.scale_tile(np.full((r, k // 32), 127, np.uint8))
    d = gpu_gemm(MX, pack(a), s(m), pack(bcodes), s(n), m, n, k, out_fp32=True)
    vals = np.array([oracle.e2m1_decode(c) for c in range(16)])
    kk = np.arange(m) * 2 % k
    expect = vals[bcodes[:, kk]].T + 2.0 * vals[bcodes[:, kk + 1]].T
    assert np.array_equal(d.astype(np.float64), expect)


# ------------------------------------------------------------ MXFP4 parity

def test_mxfp4_128x128x256_fp32_through_relayout():
    """The 128x128x256 seed-generated workload: plain scales re-laid out on the GPU."""
    w = synth.workload_inputs("mxfp4_128x128x256")
    m = n = 128
    k = 256
    sa_t = gpu_relayout(w["a_scales"], m, k, MX)
    sb_t = gpu_relayout(w["b_scales"], n, k, MX)
    d = gpu_gemm(MX, w["a_codes"], sa_t, w["b_codes"], sb_t, m, n, k, out_fp32=True)
    ref, s_abs = oracle.mx_gemm(w["a_codes"], w["a_scales"], w["b_codes"], w["b_scales"], m, n, k)
    check_fp32(d, ref, s_abs, "mxfp4 128x128x256")


@pytest.mark.parametrize("m,n,k", [(32, 32, 256), (160, 96, 512), (320, 544, 1024),
                                   (128, 256, 2048), (4000, 4064, 256), (544, 288, 768),
                                   (256, 256, 256)])
@pytest.mark.parametrize("out_fp32", [True, False])
def test_mxfp4_ragged_shapes(m, n, k, out_fp32):
    a, sa, b, sb = _codes_case(m, n, k, seed=m + n + k)
    _run_and_check_mx(a, sa, b, sb, m, n, k, out_fp32)


@pytest.mark.parametrize("split_k", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("m,n,k", [(96, 384, 2048), (288, 320, 2048)])
def test_mxfp4_explicit_split_k(split_k, m, n, k):
    """Single-CTA (M <= 128) and CTA-pair (M > 128) kernels with every split count."""
    a, sa, b, sb = _codes_case(m, n, k, seed=77)
    _run_and_check_mx(a, sa, b, sb, m, n, k, out_fp32=False, split_k=split_k)
    _run_and_check_mx(a, sa, b, sb, m, n, k, out_fp32=True, split_k=split_k)


@pytest.mark.parametrize("m,n,k,split_k", [(32, 256, 4096, 16), (64, 20480, 512, 2)])
def test_split_k_many_splits_and_many_tiles(m, n, k, split_k):
    """Split-K of the single-CTA kernel with 16 splits of one stage each, and
    with more tiles (160) than CTAs, so that a CTA takes several (tile,
    split) units in turn."""
    a, sa, b, sb = _codes_case(m, n, k, seed=79 + split_k)
    _run_and_check_mx(a, sa, b, sb, m, n, k, out_fp32=False, split_k=split_k)
    _run_and_check_mx(a, sa, b, sb, m, n, k, out_fp32=True, split_k=split_k)


@pytest.mark.parametrize("out_fp32", [True, False])
def test_split_k_tiles_do_not_depend_on_n(out_fp32):
    """The first two 128-column tiles of a 160-tile split-K GEMM (CTAs take
    several units in turn) equal, bit for bit, the same GEMM with N = 256
    (one unit per CTA): same splits, same order of the additions."""
    m, n, k = 32, 20480, 1024
    a, sa, b, sb = _codes_case(m, n, k, seed=81)
    big = gpu_gemm(MX, a, oracle.scale_tile(sa), b, oracle.scale_tile(sb), m, n, k, out_fp32,
                   split_k=2)
    small = gpu_gemm(MX, a, oracle.scale_tile(sa), b[:256], oracle.scale_tile(sb[:256]), m, 256, k,
                     out_fp32, split_k=2)
    assert np.array_equal(big[:, :256], small)
    ref, s_abs = oracle.mx_gemm(a, sa, b[:256], sb[:256], m, 256, k)
    (check_fp32 if out_fp32 else check_bf16)(small, ref, s_abs, "split 2, N = 256")


def test_single_cta_wide_tile_path():
    """M <= 128 with N wide enough for the single-CTA 256-column tile."""
    m, n, k = 96, 78848, 256
    a, sa, b, sb = _codes_case(m, n, k, seed=78)
    _run_and_check_mx(a, sa, b, sb, m, n, k, out_fp32=False, split_k=1)


@pytest.mark.parametrize("m,n,k,split_k,out_fp32", [
    (32, 2304, 4096, 1, True), (32, 2304, 4096, 3, False), (32, 640, 1024, 0, True),
    (64, 1024, 1024, 2, False), (96, 640, 768, 1, True), (32, 78848, 256, 1, False)])
def test_mxfp4_m_up_to_128_partial_a_tile(m, n, k, split_k, out_fp32):
    """The single-CTA kernel (M <= 128) loads only the M rows of A per stage and
    keeps rows M..127 of its tile at zero: M = 32, 64 and 96, with and without
    split-K, both output types, and the 256-column tile (N = 78848)."""
    a, sa, b, sb = _codes_case(m, n, k, seed=m * 7 + n + k)
    _run_and_check_mx(a, sa, b, sb, m, n, k, out_fp32, split_k=split_k)


@pytest.mark.parametrize("split_k", [0, 2])
def test_skinny_32x8192x8192_split_k_full(split_k):
    """Decode-shaped skinny GEMM split along K: every output against the oracle,
    and bit-identical across runs (fixed reduction order).  Automatic split:
    the swapped-operand kernel, whose clusters sum their partials in shared
    memory (no workspace); split_k = 2: partials in the workspace and the
    reduce kernel."""
    w = synth.workload_inputs("skinny_32x8192x8192")
    m, n, k = 32, 8192, 8192
    d1 = _run_and_check_mx(w["a_codes"], w["a_scales"], w["b_codes"], w["b_scales"], m, n, k,
                           out_fp32=False, split_k=split_k)
    d2 = gpu_gemm(MX, w["a_codes"], oracle.scale_tile(w["a_scales"]), w["b_codes"],
                  oracle.scale_tile(w["b_scales"]), m, n, k, out_fp32=False, split_k=split_k)
    assert np.array_equal(d1, d2)
    assert (mx.mx_gemm_workspace_bytes(m, n, k, split_k) > 0) == (split_k > 1)


def test_backward_gemm_with_columnwise_codes():
    """dX = dY . W through the TN GEMM: A = rowwise codes of dY [M, N], B = the
    columnwise codes of W [N, K] (the rowwise codes of W^T) from the
    bidimensional quantize; against the oracle GEMM on the oracle's codes."""
    m, n, k = 256, 512, 768
    dy = synth.bf16_normal(m, n, 1.0, seed=51)
    w = synth.bf16_normal(n, k, 0.02, seed=52)
    ca, sa_t, _ = gpu_quantize(dy, MX, TILED)
    _, _, cwt, swt = gpu_quantize_2d(w, TILED)
    ra, rsa = oracle.mx_quantize(dy)
    _, _, rwt, rswt = oracle.mx_quantize_2d(w)
    assert np.array_equal(ca, ra) and np.array_equal(cwt, rwt)
    d = gpu_gemm(MX, ca, sa_t, cwt, swt, m, k, n, out_fp32=False)
    ref, s_abs = oracle.mx_gemm(ra, rsa, rwt, rswt, m, k, n)
    check_bf16(d, ref, s_abs, "dgrad with columnwise codes")


@pytest.mark.parametrize("layout", ["TN", "NN", "TT", "NT"])
def test_four_operand_layouts_through_the_quantizer(layout):
    """D = op(A) . op(B)^T for the four layouts of BF16 inputs: an operand stored
    K-major is quantized rowwise, one stored with K as its row index
    columnwise (the bidimensional quantize, columnwise output only); the
    GEMM is the TN kernel.  Its output must equal, bit for bit, the TN GEMM
    of the explicitly transposed inputs, and match the oracle."""
    m, n, k = 160, 288, 512
    a_km = synth.bf16_normal(m, k, 1.0, seed=61)          # A as [M, K]
    b_kn = synth.bf16_normal(n, k, 0.05, seed=62)         # B as [N, K]
    # A is stored [M, K] for TN and NN, [K, M] for TT and NT; B [N, K] for TN and TT, [K, N] otherwise
    a_stored = a_km if layout in ("TN", "NN") else np.ascontiguousarray(a_km.T)
    b_stored = b_kn if layout in ("TN", "TT") else np.ascontiguousarray(b_kn.T)

    def k_major(x_stored, is_k_major):
        if is_k_major:
            c, s_t, _ = gpu_quantize(x_stored, MX, TILED)
            return c, s_t
        _, _, ct, st = gpu_quantize_2d(x_stored, TILED, columnwise_only=True)
        return ct, st
    ca, sa = k_major(a_stored, layout in ("TN", "NN"))
    cb, sb = k_major(b_stored, layout in ("TN", "TT"))
    d = gpu_gemm(MX, ca, sa, cb, sb, m, n, k, out_fp32=False)
    ra, rsa = oracle.mx_quantize(a_km)
    rb, rsb = oracle.mx_quantize(b_kn)
    assert np.array_equal(ca, ra) and np.array_equal(cb, rb)
    d_tn = gpu_gemm(MX, ra, oracle.scale_tile(rsa), rb, oracle.scale_tile(rsb), m, n, k,
                    out_fp32=False)
    assert np.array_equal(d, d_tn)
    ref, s_abs = oracle.mx_gemm(ra, rsa, rb, rsb, m, n, k)
    check_bf16(d, ref, s_abs, f"layout {layout}")


# ------------------------------------------------------------ FP4 code transpose

def _gpu_transpose(codes, rows, cols):
    out = guarded(rows * cols // 2, fill=0xAB)
    mx.mx_fp4_transpose(dev_u8(codes), rows, cols, out)
    torch.cuda.synchronize()
    check_guards(out, what=f"FP4 transpose {rows}x{cols}")
    return out.cpu().numpy().reshape(cols, rows // 2)


@pytest.mark.parametrize("rows,cols", [(32, 32), (64, 128), (96, 4128), (160, 96), (4096, 1056),
                                       (8192, 8192), (1 << 21, 64), (32, 1 << 22)])
def test_fp4_transpose_matches_oracle(rows, cols):
    """Bit-exact against the oracle: one and several 128 x 256 tiles, ragged
    tails in both directions, a full 8192 x 8192 weight, and tile grids 16384
    tiles tall or 16384 tiles wide."""
    codes = synth.fp4_codes(rows, cols, seed=rows * 7 + cols)
    assert np.array_equal(_gpu_transpose(codes, rows, cols),
                          oracle.fp4_transpose(codes, rows, cols))


def test_fp4_transpose_workload_full_size():
    """The transpose workload as bench.py runs it (the MLP weight's codes
    stored 8192 x 28672), every byte."""
    name = "fp4_transpose_8192x28672"
    wl = synth.WORKLOADS[name]
    codes = synth.workload_inputs(name)["a_codes"]
    assert np.array_equal(_gpu_transpose(codes, wl["m"], wl["k"]),
                          oracle.fp4_transpose(codes, wl["m"], wl["k"]))


@pytest.mark.parametrize("stored_mn", ["A", "B", "AB"])
def test_gemm_of_operands_stored_mn_contiguous(stored_mn):
    """Operands quantized along K but stored M- or N-contiguous (the NN, NT and
    TT layouts): the GPU transpose brings them to K-contiguous codes, equal to
    the original ones, and the TN GEMM then gives the same bits as on the
    original operands, within the tolerances of the oracle."""
    m, n, k = 160, 288, 512
    a, sa, b, sb = _codes_case(m, n, k, seed=77)
    a_in = oracle.fp4_transpose(a, m, k) if "A" in stored_mn else a      # [K, M/2] when stored MN
    b_in = oracle.fp4_transpose(b, n, k) if "B" in stored_mn else b
    a_km = _gpu_transpose(a_in, k, m) if "A" in stored_mn else a_in
    b_km = _gpu_transpose(b_in, k, n) if "B" in stored_mn else b_in
    assert np.array_equal(a_km, a) and np.array_equal(b_km, b)
    d = gpu_gemm(MX, a_km, oracle.scale_tile(sa), b_km, oracle.scale_tile(sb), m, n, k, True)
    d_tn = gpu_gemm(MX, a, oracle.scale_tile(sa), b, oracle.scale_tile(sb), m, n, k, True)
    assert np.array_equal(d.view(np.uint32), d_tn.view(np.uint32))
    ref, s_abs = oracle.mx_gemm(a, sa, b, sb, m, n, k)
    check_fp32(d, ref, s_abs, f"operands stored MN-contiguous: {stored_mn}")


def _quant_gemm_check(name, n_rows, n_cols):
    wl = synth.WORKLOADS[name]
    m, n, k = wl["m"], wl["n"], wl["k"]
    w = synth.workload_inputs(name)
    ca, sa_t, _ = gpu_quantize(w["a"], MX, TILED)
    cb, sb_t, _ = gpu_quantize(w["b"], MX, TILED)
    ra, rsa = oracle.mx_quantize(w["a"])
    rb, rsb = oracle.mx_quantize(w["b"])
    assert np.array_equal(ca, ra) and np.array_equal(cb, rb)
    del w
    out_fp32 = wl["out"] == "fp32"
    check = check_fp32 if out_fp32 else check_bf16
    d = gpu_gemm(MX, ca, sa_t, cb, sb_t, m, n, k, out_fp32=out_fp32)
    rows = sample_indices(m, n_rows, 128, seed=1)
    cols = sample_indices(n, n_cols, 256, seed=2)
    ref, s_abs = oracle.mx_gemm(ra, rsa, rb, rsb, m, n, k, rows=rows)
    st = check(d[rows], ref, s_abs, f"{name} sampled rows")
    ref, s_abs = oracle.mx_gemm(ra, rsa, rb, rsb, m, n, k, cols=cols)
    check(d[:, cols], ref, s_abs, f"{name} sampled cols")
    assert np.count_nonzero(d) > 0.99 * d.size
    return st


def test_quant_gemm_2048x4096x4096_bf16():
    _quant_gemm_check("quant_gemm_2048x4096x4096", 96, 64)


def test_mlp_up_16384x28672x8192_bf16_sampled():
    _quant_gemm_check("mlp_up_16384x28672x8192", 32, 24)


def test_mxfp4_4096_cubed_fp32_sampled():
    _quant_gemm_check("mxfp4_4096x4096x4096", 96, 64)


# ------------------------------------------------------------ NVFP4 parity

@pytest.mark.parametrize("m,n,k,split_k", [(128, 128, 256, 1), (256, 320, 1024, 1),
                                           (160, 4096, 512, 1), (64, 512, 2048, 3),
                                           (416, 352, 2048, 3), (32, 640, 1024, 1),
                                           (32, 640, 1024, 3)])
def test_nvfp4_gemm_small(m, n, k, split_k):
    xa = synth.bf16_normal(m, k, 1.0, seed=m * 3 + k)
    xb = synth.bf16_normal(n, k, 1.0, seed=n * 5 + k)
    ca, sa_t, ta = gpu_quantize(xa, NV, TILED)
    cb, sb_t, tb = gpu_quantize(xb, NV, TILED)
    ra, rsa, rta = oracle.nvfp4_quantize(xa)
    rb, rsb, rtb = oracle.nvfp4_quantize(xb)
    assert np.array_equal(ca, ra) and np.array_equal(cb, rb) and ta == rta and tb == rtb
    d = gpu_gemm(NV, ca, sa_t, cb, sb_t, m, n, k, out_fp32=True, split_k=split_k, a_ts=ta, b_ts=tb)
    ref, s_abs = oracle.nvfp4_gemm(ra, rsa, rb, rsb, m, n, k, rta, rtb)
    check_fp32(d, ref, s_abs, f"nvfp4 {m}x{n}x{k}")


def test_nvfp4_4096_cubed_fp32_sampled():
    name = "nvfp4_4096x4096x4096"
    m = n = k = 4096
    w = synth.workload_inputs(name)
    ca, sa_t, ta = gpu_quantize(w["a"], NV, TILED)
    cb, sb_t, tb = gpu_quantize(w["b"], NV, TILED)
    ra, rsa, rta = oracle.nvfp4_quantize(w["a"])
    rb, rsb, rtb = oracle.nvfp4_quantize(w["b"])
    d = gpu_gemm(NV, ca, sa_t, cb, sb_t, m, n, k, out_fp32=True, a_ts=ta, b_ts=tb)
    rows = sample_indices(m, 96, 128, seed=3)
    cols = sample_indices(n, 64, 256, seed=4)
    ref, s_abs = oracle.nvfp4_gemm(ra, rsa, rb, rsb, m, n, k, rta, rtb, rows=rows)
    check_fp32(d[rows], ref, s_abs, "nvfp4 4096^3 rows")
    ref, s_abs = oracle.nvfp4_gemm(ra, rsa, rb, rsb, m, n, k, rta, rtb, cols=cols)
    check_fp32(d[:, cols], ref, s_abs, "nvfp4 4096^3 cols")


# ------------------------------------------------------------ contract on the GPU

def test_workspace_too_small_is_rejected():
    m, n, k = 32, 1024, 4096
    a, sa, b, sb = _codes_case(m, n, k, seed=5)
    d = torch.full((m, n), 7.0, dtype=torch.float32, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(mx.MXError) as e:
        mx.mxfp4_gemm(dev_u8(a), dev_u8(oracle.scale_tile(sa)), dev_u8(b),
                      dev_u8(oracle.scale_tile(sb)), d, m, n, k, mx.MX_LAYOUT_TN, mx.MX_OUT_FP32,
                      4, ws)
    assert e.value.code == mx.MX_ERR_WORKSPACE
    torch.cuda.synchronize()
    assert torch.all(d == 7.0)           # nothing written on an argument error


def test_device_is_available():
    assert mx.mx_available()


def test_pair_gemm_very_tall_a():
    """M = 2^17 rows of A (512 256-row tiles, 6.7 waves of pair tiles), N = 256,
    K = 256: the tile walk and the output offsets at a size where 32-bit products
    of them would overflow; every output against the oracle."""
    m, n, k = 1 << 17, 256, 256
    a = synth.fp4_codes(m, k, 91)
    sa = synth.scale_bytes(m, k // 32, 120, 134, 92)
    b = synth.fp4_codes(n, k, 93)
    sb = synth.scale_bytes(n, k // 32, 120, 134, 94)
    d = gpu_gemm(MX, a, oracle.scale_tile(sa), b, oracle.scale_tile(sb), m, n, k, out_fp32=False)
    ref, s_abs = oracle.mx_gemm(a, sa, b, sb, m, n, k)
    stats = check_bf16(d, ref, s_abs, "pair 2^17 x 256 x 256")
    assert stats["exact"] > 0.9 * stats["total"]
