"""GPU parity of the GEMM epilogue (bias, beta * D_in, GELU) against the oracle.

The oracle gives act(alpha A B^T + beta C + bias) in binary64.  The kernel
takes the FP32 accumulator through one binary32 operation per term and its
own GELU, then rounds once to the output type, so an output passes
when it is within
    E = L * (E_acc + 2^-22 (|alpha A B^T| + |beta C| + |bias| + |y|))
        + (GELU: the GELU term below)
of the oracle's value (FP32 out), or within E plus one BF16 ulp (BF16 out),
where the GELU term is |GELU(y)| 2^-24 * 44, the error bound of the kernel's
GELU (a Chebyshev fit of erfc with fractional error below 1.2e-7, CUDA's expf
and fast reciprocal at 2 ulp each, the Horner and product roundings; the
rounding of the exponent argument, of magnitude up to y^2 / 2, is recovered
exactly and applied as a first-order correction, so it adds no y^2 term).  E_acc is the accumulation bound of the plain GEMM tests (1e-5
sum |a||b|), L = 1.13 >= max |GELU'| with GELU and 1 without it, and 2^-22
covers one rounding of each of the (at most three) binary32 steps.
"""
import numpy as np
import pytest
import torch

import block_scaled_fp4_bf16_gb300 as mx
import oracle
from block_scaled_fp4_bf16_gb300 import synth
from tests.gpu_helpers import (FP32_REL_TOL, bf16_bits_to_f64, check_guards, dev_u8, gpu_quantize,
                               guarded)

pytestmark = pytest.mark.gpu

MX, NV = mx.MX_FMT_MXFP4, mx.MX_FMT_NVFP4
TILED = mx.MX_SCALE_TCGEN05


def _bf16_ulp_at(v):
    """BF16 spacing at magnitude |v| (fp64)."""
    a = np.maximum(np.abs(v), 2.0 ** -133)
    e = np.floor(np.log2(a))
    return np.maximum(2.0 ** (e - 7), 2.0 ** -133)


def _run(fmt, ops, m, n, k, out_fp32, split_k, bias, beta, gelu, d_in):
    """GEMM with an epilogue; d_in: host values D holds before the call (or None: NaN)."""
    dt = torch.float32 if out_fp32 else torch.bfloat16
    body = guarded(m * n, dt, float("nan"))
    d = body.view(m, n)
    d._mx_guard = body._mx_guard
    if d_in is not None:
        d.copy_(torch.from_numpy(np.asarray(d_in, np.float32)).to("cuda").to(dt))
    b = None if bias is None else torch.from_numpy(np.asarray(bias, np.float32)).to("cuda")
    wsb = mx.mx_gemm_workspace_bytes(m, n, k, split_k)
    ws = guarded(max(wsb, 16)) if wsb else None
    od = mx.MX_OUT_FP32 if out_fp32 else mx.MX_OUT_BF16
    if fmt == MX:
        a, sa, bb, sb = ops
        mx.mxfp4_gemm_ex(dev_u8(a), dev_u8(sa), dev_u8(bb), dev_u8(sb), d, m, n, k,
                         mx.MX_LAYOUT_TN, od, split_k, b, beta, gelu, ws)
    else:
        a, sa, bb, sb, ta, tb = ops
        tat = torch.tensor([ta], dtype=torch.float32, device="cuda")
        tbt = torch.tensor([tb], dtype=torch.float32, device="cuda")
        mx.nvfp4_gemm_ex(dev_u8(a), dev_u8(sa), dev_u8(bb), dev_u8(sb), tat, tbt, d, m, n, k,
                         mx.MX_LAYOUT_TN, od, split_k, b, beta, gelu, ws)
    torch.cuda.synchronize()
    assert mx.mx_device_status() == mx.MX_OK
    check_guards(d, ws, what=f"GEMM epilogue {m}x{n}x{k} split {split_k}")
    if out_fp32:
        return d.cpu().numpy().astype(np.float64)
    return bf16_bits_to_f64(d.view(torch.int16).cpu().numpy().view(np.uint16))


def _check(got, d_ref, s_abs, bias, beta, c, gelu, out_fp32, what):
    y = oracle.gemm_epilogue(d_ref, bias=bias, gelu_on=False, beta=beta,
                             c=None if c is None or beta == 0 else c)
    ref = oracle.gemm_epilogue(d_ref, bias=bias, gelu_on=gelu, beta=beta,
                               c=None if c is None or beta == 0 else c)
    terms = np.abs(d_ref) + np.abs(y)
    if c is not None and beta != 0:
        terms = terms + np.abs(beta * c)
    if bias is not None:
        terms = terms + np.abs(np.asarray(bias, np.float64))[None, :]
    lip = 1.13 if gelu else 1.0
    e = lip * (FP32_REL_TOL * s_abs + 2.0 ** -22 * terms)
    if gelu:
        e = e + 2.0 ** -24 * 44 * np.abs(ref)
    if not out_fp32:
        e = e + _bf16_ulp_at(np.abs(ref) + e)
    e = e + 1e-30
    assert np.all(np.isfinite(got)), f"{what}: non-finite outputs"
    bad = np.abs(got - ref) > e
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())}/{bad.size} outputs out of tolerance; first "
                             + ", ".join(f"{tuple(x)} got {got[tuple(x)]!r} ref {ref[tuple(x)]!r} "
                                         f"tol {e[tuple(x)]!r}" for x in i))


def _mx_case(m, n, k, seed):
    # scales near 2^-3 keep the products O(1): y spans the whole GELU range
    a = synth.fp4_codes(m, k, seed)
    sa = synth.scale_bytes(m, k // 32, 122, 126, seed + 1)
    b = synth.fp4_codes(n, k, seed + 2)
    sb = synth.scale_bytes(n, k // 32, 122, 126, seed + 3)
    ref, s_abs = oracle.mx_gemm(a, sa, b, sb, m, n, k)
    return (a, oracle.scale_tile(sa), b, oracle.scale_tile(sb)), ref, s_abs


def _inputs(ref, n, seed, out_fp32):
    rng = np.random.default_rng(seed)
    sd = float(np.std(ref)) or 1.0
    bias = (rng.standard_normal(n) * sd).astype(np.float32)
    c = (rng.standard_normal(ref.shape) * sd).astype(np.float32)
    if not out_fp32:  # D_in is held in BF16: the reference uses the stored values
        c = synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(c))
    return bias, c.astype(np.float64)


# (m, n, k, split_k): the CTA-pair kernel, the single-CTA kernel, split-K, and
# the swapped-operand kernel for M <= 64 (automatic split: one CTA, and a
# cluster of CTAs whose partials meet in shared memory)
SHAPES = [(256, 512, 1024, 1), (96, 384, 512, 1), (96, 384, 2048, 3), (320, 288, 1024, 2),
          (32, 640, 1024, 0), (64, 4224, 4096, 0), (32, 20480, 512, 0)]
# (bias, beta, gelu)
TERMS = [(True, 0.0, False), (False, 0.0, True), (True, 0.0, True), (False, 1.0, False),
         (True, 0.5, True), (True, -2.0, False)]


@pytest.mark.parametrize("m,n,k,split_k", SHAPES)
@pytest.mark.parametrize("out_fp32", [True, False])
@pytest.mark.parametrize("use_bias,beta,gelu", TERMS)
def test_mxfp4_epilogue_matches_oracle(m, n, k, split_k, out_fp32, use_bias, beta, gelu):
    ops, ref, s_abs = _mx_case(m, n, k, seed=m + n + k)
    bias, c = _inputs(ref, n, seed=7, out_fp32=out_fp32)
    bias = bias if use_bias else None
    got = _run(MX, ops, m, n, k, out_fp32, split_k, bias, beta, gelu,
               c if beta != 0 else None)
    _check(got, ref, s_abs, bias, beta, c, gelu, out_fp32,
           f"mxfp4 {m}x{n}x{k} split {split_k} fp32={out_fp32} bias={use_bias} beta={beta} gelu={gelu}")


@pytest.mark.parametrize("m,n,k,split_k", [(256, 320, 1024, 1), (64, 512, 2048, 3), (32, 640, 1024, 1),
                                           (32, 4096, 4096, 0)])
@pytest.mark.parametrize("out_fp32", [True, False])
def test_nvfp4_epilogue_matches_oracle(m, n, k, split_k, out_fp32):
    xa = synth.bf16_normal(m, k, 1.0, seed=m * 3 + k)
    xb = synth.bf16_normal(n, k, 0.05, seed=n * 5 + k)
    ca, sa_t, ta = gpu_quantize(xa, NV, TILED)
    cb, sb_t, tb = gpu_quantize(xb, NV, TILED)
    ra, rsa, rta = oracle.nvfp4_quantize(xa)
    rb, rsb, rtb = oracle.nvfp4_quantize(xb)
    assert np.array_equal(ca, ra) and np.array_equal(cb, rb)
    ref, s_abs = oracle.nvfp4_gemm(ra, rsa, rb, rsb, m, n, k, rta, rtb)
    bias, c = _inputs(ref, n, seed=8, out_fp32=out_fp32)
    got = _run(NV, (ca, sa_t, cb, sb_t, ta, tb), m, n, k, out_fp32, split_k, bias, 0.75, True, c)
    _check(got, ref, s_abs, bias, 0.75, c, True, out_fp32, f"nvfp4 {m}x{n}x{k} split {split_k}")


def test_beta_zero_keeps_d_write_only():
    """With a bias and GELU but beta == 0 a NaN-filled D must not leak into the output."""
    m, n, k = 256, 256, 512
    ops, ref, s_abs = _mx_case(m, n, k, seed=3)
    bias, _ = _inputs(ref, n, seed=9, out_fp32=True)
    got = _run(MX, ops, m, n, k, True, 1, bias, 0.0, True, None)
    _check(got, ref, s_abs, bias, 0.0, None, True, True, "beta 0")


def test_accumulate_twice_into_fp32():
    """D = A B^T + 1 * D run twice from D = 0 gives 2 A B^T (gradient accumulation)."""
    m, n, k = 128, 384, 1024
    ops, ref, s_abs = _mx_case(m, n, k, seed=4)
    a, sa, b, sb = ops
    d = torch.zeros((m, n), dtype=torch.float32, device="cuda")
    for _ in range(2):
        mx.mxfp4_gemm_ex(dev_u8(a), dev_u8(sa), dev_u8(b), dev_u8(sb), d, m, n, k, mx.MX_LAYOUT_TN,
                         mx.MX_OUT_FP32, 1, None, 1.0, False, None)
    torch.cuda.synchronize()
    got = d.cpu().numpy().astype(np.float64)
    tol = 2 * FP32_REL_TOL * s_abs + 2.0 ** -22 * np.abs(2 * ref) + 1e-30
    assert np.all(np.abs(got - 2 * ref) <= tol)


def test_plain_entry_points_unchanged_by_a_null_epilogue():
    """mxfp4_gemm_ex with no terms is the plain GEMM, bit for bit."""
    m, n, k = 256, 512, 1024
    ops, _, _ = _mx_case(m, n, k, seed=5)
    a, sa, b, sb = ops
    out = []
    for ex in (False, True):
        d = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        if ex:
            mx.mxfp4_gemm_ex(dev_u8(a), dev_u8(sa), dev_u8(b), dev_u8(sb), d, m, n, k,
                             mx.MX_LAYOUT_TN, mx.MX_OUT_BF16, 0)
        else:
            mx.mxfp4_gemm(dev_u8(a), dev_u8(sa), dev_u8(b), dev_u8(sb), d, m, n, k,
                          mx.MX_LAYOUT_TN, mx.MX_OUT_BF16, 0)
        torch.cuda.synchronize()
        out.append(d.view(torch.int16).cpu().numpy())
    assert np.array_equal(out[0], out[1])


def test_bias_gelu_workload_full_size_sampled():
    """The bias + GELU workload as bench.py runs it (quantize A and W, GEMM with
    the FP32 bias and GELU), checked on sampled output rows."""
    from tests.gpu_helpers import sample_indices
    name = "quant_gemm_bias_gelu_2048x4096x4096"
    w = synth.workload_inputs(name)
    m, n, k = 2048, 4096, 4096
    ca, sa_t, _ = gpu_quantize(w["a"], MX, TILED)
    cb, sb_t, _ = gpu_quantize(w["b"], MX, TILED)
    ra, rsa = oracle.mx_quantize(w["a"])
    rb, rsb = oracle.mx_quantize(w["b"])
    assert np.array_equal(ca, ra) and np.array_equal(cb, rb)
    got = _run(MX, (ca, sa_t, cb, sb_t), m, n, k, False, 1, w["bias"], 0.0, True, None)
    rows = sample_indices(m, 48, 256, seed=11)
    ref, s_abs = oracle.mx_gemm(ra, rsa, rb, rsb, m, n, k, rows=rows)
    _check(got[rows], ref, s_abs, w["bias"], 0.0, None, True, False, "bias+gelu workload")
