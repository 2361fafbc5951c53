"""mxfp4_gemm_static_workspace: the MXFP4 GEMM for callers that cannot allocate
device memory (a plugin in a host program that owns all device memory, or a path
where a new allocation is not allowed).  Its split-K scratch is a fixed array in
the library instead of a caller-provided workspace.

Checked through the C ABI on calls in a row that all use the shared scratch:
each result is bit-identical to mxfp4_gemm with a caller workspace (the same
kernels and the same fixed split order, so any stale or missed partial would
show as a changed bit), and within the tolerances of the other GEMM tests of
the oracle's D (FP32: 1e-5 * sum |a||b|; BF16: 1 ulp of the correctly rounded
value).  This file is collected last, and passes both alone in a fresh process
and after the other tests.
"""
import numpy as np
import pytest
import torch

import block_scaled_fp4_bf16_gb300 as mx
import oracle
from block_scaled_fp4_bf16_gb300 import synth
from tests.gpu_helpers import check_bf16, check_fp32, dev_u8

pytestmark = pytest.mark.gpu


def _inputs(m, n, k, seed):
    a = synth.fp4_codes(m, k, seed)
    b = synth.fp4_codes(n, k, seed + 1)
    sa = synth.scale_bytes(m, k // 32, 122, 130, seed + 2)
    sb = synth.scale_bytes(n, k // 32, 122, 130, seed + 3)
    return a, sa, b, sb


def _bits(d: torch.Tensor) -> np.ndarray:
    """The raw bits of a device result (NaN-safe comparison)."""
    if d.dtype == torch.float32:
        return d.view(torch.int32).cpu().numpy().view(np.uint32)
    return d.view(torch.int16).cpu().numpy().view(np.uint16)


def _run_both(a, sa, b, sb, m, n, k, split_k, out_dtype):
    """Returns the bits of (static-scratch result, workspace result)."""
    da, dsa = dev_u8(a), dev_u8(oracle.scale_tile(sa))
    db, dsb = dev_u8(b), dev_u8(oracle.scale_tile(sb))
    dt = torch.float32 if out_dtype == mx.MX_OUT_FP32 else torch.bfloat16
    d_static = torch.full((m, n), float("nan"), dtype=dt, device="cuda")
    d_ws = torch.full((m, n), float("nan"), dtype=dt, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = mx.lib().mxfp4_gemm_static_workspace(
        da.data_ptr(), dsa.data_ptr(), db.data_ptr(), dsb.data_ptr(), d_static.data_ptr(),
        m, n, k, mx.MX_LAYOUT_TN, out_dtype, split_k, stream)
    assert rc == mx.MX_OK, mx.mx_last_error_string()
    wsb = mx.mx_gemm_workspace_bytes(m, n, k, split_k)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    rc = mx.lib().mxfp4_gemm(
        da.data_ptr(), dsa.data_ptr(), db.data_ptr(), dsb.data_ptr(), d_ws.data_ptr(),
        m, n, k, mx.MX_LAYOUT_TN, out_dtype, split_k, ws.data_ptr(), wsb, stream)
    assert rc == mx.MX_OK, mx.mx_last_error_string()
    torch.cuda.synchronize()
    assert mx.mx_device_status() == mx.MX_OK
    return _bits(d_static), _bits(d_ws)


def test_static_workspace_matches_workspace_gemm_and_oracle_on_calls_in_a_row():
    # the decode-shaped skinny GEMM with two and four splits, an explicit split
    # count on other data, and the automatic split of M = 96: calls in a row that
    # all use the shared scratch, each leaving partials the next must not read.
    # (M <= 64 with the automatic split needs no scratch: its partial sums meet
    # in shared memory.)
    cases = [(32, 8192, 8192, 2, 401, mx.MX_OUT_BF16),
             (64, 1024, 4096, 4, 402, mx.MX_OUT_FP32),
             (96, 2048, 2048, 0, 403, mx.MX_OUT_BF16),
             (32, 8192, 8192, 4, 404, mx.MX_OUT_FP32)]
    for m, n, k, split_k, seed, out in cases:
        need = mx.mx_gemm_workspace_bytes(m, n, k, split_k)
        assert 0 < need <= mx.MX_STATIC_WORKSPACE_BYTES      # split-K really runs
        a, sa, b, sb = _inputs(m, n, k, seed)
        d_static, d_ws = _run_both(a, sa, b, sb, m, n, k, split_k, out)
        what = f"static scratch {m}x{n}x{k} split {split_k}"
        assert np.array_equal(d_static, d_ws), f"{what}: differs from the workspace GEMM"
        ref, s_abs = oracle.mx_gemm(a, sa, b, sb, m, n, k)
        if out == mx.MX_OUT_FP32:
            check_fp32(d_static.view(np.float32), ref, s_abs, what)
        else:
            check_bf16(d_static, ref, s_abs, what)


def test_static_workspace_rejects_shapes_beyond_its_size():
    m, n, k, split_k = 1024, 4096, 4096, 2
    assert mx.mx_gemm_workspace_bytes(m, n, k, split_k) > mx.MX_STATIC_WORKSPACE_BYTES
    a = torch.zeros(m * k // 2, dtype=torch.uint8, device="cuda")
    b = torch.zeros(n * k // 2, dtype=torch.uint8, device="cuda")
    sa = torch.zeros(mx.mx_scale_bytes(m, k, 0, 1), dtype=torch.uint8, device="cuda")
    sb = torch.zeros(mx.mx_scale_bytes(n, k, 0, 1), dtype=torch.uint8, device="cuda")
    d = torch.full((m, n), 7.0, dtype=torch.float32, device="cuda")
    with pytest.raises(mx.MXError) as e:
        mx.mxfp4_gemm_static_workspace(a, sa, b, sb, d, m, n, k, mx.MX_LAYOUT_TN,
                                       mx.MX_OUT_FP32, split_k)
    assert e.value.code == mx.MX_ERR_WORKSPACE
    assert "more than the 16777216 bytes of the static array" in e.value.detail
    torch.cuda.synchronize()
    assert torch.all(d == 7.0)   # rejected before anything was launched
