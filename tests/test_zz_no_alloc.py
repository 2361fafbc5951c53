"""mxfp4_gemm_static_workspace: the MXFP4 GEMM for callers that cannot allocate
device memory (a plugin in a host program that owns all device memory, or a path
where a new allocation is not allowed).  Its split-K scratch is a fixed array in
the library instead of a caller-provided workspace.

Checked through the C ABI against mxfp4_gemm with a workspace, on two calls in a
row, within the FP32 tolerance of the other GEMM tests.  This file is collected
last, and passes both alone in a fresh process and after the other tests.
"""
import numpy as np
import pytest
import torch

import block_scaled_fp4_bf16_gb300 as mx
import oracle
from block_scaled_fp4_bf16_gb300 import synth
from tests.gpu_helpers import check_fp32, dev_u8

pytestmark = pytest.mark.gpu


def _inputs(m, n, k, seed):
    a = synth.fp4_codes(m, k, seed)
    b = synth.fp4_codes(n, k, seed + 1)
    sa = synth.scale_bytes(m, k // 32, 122, 130, seed + 2)
    sb = synth.scale_bytes(n, k // 32, 122, 130, seed + 3)
    return a, sa, b, sb


def _run_both(a, sa, b, sb, m, n, k, split_k):
    """Returns (static-scratch result, workspace result) as host FP32 arrays."""
    da, dsa = dev_u8(a), dev_u8(oracle.scale_tile(sa))
    db, dsb = dev_u8(b), dev_u8(oracle.scale_tile(sb))
    d_static = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    d_ws = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = mx.lib().mxfp4_gemm_static_workspace(
        da.data_ptr(), dsa.data_ptr(), db.data_ptr(), dsb.data_ptr(), d_static.data_ptr(),
        m, n, k, mx.MX_LAYOUT_TN, mx.MX_OUT_FP32, split_k, stream)
    assert rc == mx.MX_OK, mx.mx_error_string(rc)
    wsb = mx.mx_gemm_workspace_bytes(m, n, k, split_k)
    ws = torch.empty(wsb, dtype=torch.uint8, device="cuda")
    rc = mx.lib().mxfp4_gemm(
        da.data_ptr(), dsa.data_ptr(), db.data_ptr(), dsb.data_ptr(), d_ws.data_ptr(),
        m, n, k, mx.MX_LAYOUT_TN, mx.MX_OUT_FP32, split_k, ws.data_ptr(), wsb, stream)
    assert rc == mx.MX_OK, mx.mx_error_string(rc)
    torch.cuda.synchronize()
    assert mx.mx_device_status() == mx.MX_OK
    return d_static.cpu().numpy(), d_ws.cpu().numpy()


def test_static_workspace_matches_workspace_gemm_twice():
    # the decode-shaped skinny GEMM (automatic split-K), then an explicit split
    # count on other data: two calls in a row that both use the shared scratch
    for m, n, k, split_k, seed in [(32, 8192, 8192, 0, 401), (64, 1024, 4096, 4, 402)]:
        need = mx.mx_gemm_workspace_bytes(m, n, k, split_k)
        assert 0 < need <= mx.MX_STATIC_WORKSPACE_BYTES      # split-K really runs
        a, sa, b, sb = _inputs(m, n, k, seed)
        d_static, d_ws = _run_both(a, sa, b, sb, m, n, k, split_k)
        _, s_abs = oracle.mx_gemm(a, sa, b, sb, m, n, k)
        check_fp32(d_static, d_ws.astype(np.float64), s_abs, f"static scratch {m}x{n}x{k}")


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
    torch.cuda.synchronize()
    assert torch.all(d == 7.0)   # rejected before anything was launched
