"""The C-ABI library loads and exports every entry point of include/mxfp4.h, and
its host-side contract (sizes, error strings, argument validation) holds.  No
call here reaches the GPU: validation rejects each call before any device
work, and the library never dereferences the fake pointers used below."""
import ctypes
import os
import re

import pytest

import block_scaled_fp4_bf16_gb300 as mx

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxfp4.h")


@pytest.fixture(scope="module")
def lib():
    from block_scaled_fp4_bf16_gb300 import build
    build.build()
    return mx.lib()


def _declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mx\w+|mxfp4_\w+|nvfp4_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ["mx_quantize_bf16", "mxfp4_gemm", "nvfp4_gemm", "mx_scale_relayout",
                     "mx_device_status", "mx_error_string", "mx_available"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in _declared_functions():
        assert hasattr(lib, name), name
        assert isinstance(getattr(lib, name), ctypes._CFuncPtr)


def test_error_strings(lib):
    codes = [0, -1, -2, -3, -4, -5, -6, -7, -8, -9, -10]
    texts = [mx.mx_error_string(c) for c in codes]
    assert len(set(texts)) == len(codes)
    assert mx.mx_error_string(-100) == "unknown status code"


def test_scale_bytes(lib):
    assert mx.mx_scale_bytes(128, 256, mx.MX_FMT_MXFP4, mx.MX_SCALE_PLAIN) == 128 * 8
    assert mx.mx_scale_bytes(128, 256, mx.MX_FMT_MXFP4, mx.MX_SCALE_TCGEN05) == 128 * 8
    assert mx.mx_scale_bytes(32, 256, mx.MX_FMT_MXFP4, mx.MX_SCALE_TCGEN05) == 128 * 8
    assert mx.mx_scale_bytes(200, 96, mx.MX_FMT_MXFP4, mx.MX_SCALE_TCGEN05) == 256 * 4
    assert mx.mx_scale_bytes(16384, 8192, mx.MX_FMT_MXFP4, mx.MX_SCALE_TCGEN05) == 16384 * 256
    assert mx.mx_scale_bytes(4096, 4096, mx.MX_FMT_NVFP4, mx.MX_SCALE_TCGEN05) == 4096 * 256
    assert mx.mx_scale_bytes(4096, 4096, mx.MX_FMT_NVFP4, mx.MX_SCALE_PLAIN) == 4096 * 256
    assert mx.mx_scale_bytes(4, 33, mx.MX_FMT_MXFP4, mx.MX_SCALE_PLAIN) == 0
    assert mx.mx_scale_bytes(4, 32, 7, mx.MX_SCALE_PLAIN) == 0
    assert mx.mx_scale_bytes(0, 32, mx.MX_FMT_MXFP4, mx.MX_SCALE_PLAIN) == 0


def test_workspace_bytes(lib):
    assert mx.mx_quantize_workspace_bytes(10, 32, mx.MX_FMT_MXFP4) == 0
    assert mx.mx_quantize_workspace_bytes(10, 32, mx.MX_FMT_NVFP4) > 0
    assert mx.mx_gemm_workspace_bytes(4096, 4096, 4096, 1) == 0
    assert mx.mx_gemm_workspace_bytes(32, 8192, 8192, 4) == 4 * 32 * 8192 * 4
    assert mx.mx_gemm_workspace_bytes(32, 8192, 8192, 0) % (32 * 8192 * 4) == 0
    assert mx.mx_gemm_workspace_bytes(32, 8192, 100, 1) == 0  # K % 256 != 0


FAKE = 1 << 40        # a 16-byte aligned address that is never dereferenced
FAKE_ODD = FAKE + 8   # not 16-byte aligned


def _gemm(lib, **kw):
    a = dict(a=FAKE, sa=FAKE, b=FAKE, sb=FAKE, d=FAKE, m=128, n=128, k=256, layout=0, out=0,
             split=1, ws=None, wsb=0)
    a.update(kw)
    return lib.mxfp4_gemm(a["a"], a["sa"], a["b"], a["sb"], a["d"], a["m"], a["n"], a["k"],
                          a["layout"], a["out"], a["split"], a["ws"], a["wsb"], None)


def test_gemm_argument_validation(lib):
    assert _gemm(lib, a=None) == mx.MX_ERR_INVALID_ARG
    assert _gemm(lib, d=None) == mx.MX_ERR_INVALID_ARG
    assert _gemm(lib, split=-1) == mx.MX_ERR_INVALID_ARG
    assert _gemm(lib, layout=1) == mx.MX_ERR_UNSUPPORTED_FEATURE
    assert _gemm(lib, out=2) == mx.MX_ERR_UNSUPPORTED_FEATURE
    assert _gemm(lib, k=128) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert _gemm(lib, m=48) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert _gemm(lib, n=40) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert _gemm(lib, m=0) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert _gemm(lib, a=FAKE_ODD) == mx.MX_ERR_ALIGNMENT
    assert _gemm(lib, d=FAKE_ODD) == mx.MX_ERR_ALIGNMENT
    # NVFP4 needs both tensor scales
    assert lib.nvfp4_gemm(FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, 128, 128, 256, 0, 1, 1,
                          None, 0, None) == mx.MX_ERR_INVALID_ARG


def test_gemm_epilogue_argument_validation(lib):
    MB = 1 << 20

    def call(gelu=0, bias=None, beta=0.0, d=FAKE + 4 * MB, m=128, n=128):
        ep = mx.mx_gemm_epilogue(bias, beta, gelu)
        return lib.mxfp4_gemm_ex(FAKE, FAKE + MB, FAKE + 2 * MB, FAKE + 3 * MB, d, m, n, 256, 0, 0, 1,
                                 ctypes.byref(ep), None, 0, None)
    assert call(gelu=2) == mx.MX_ERR_INVALID_ARG
    assert call(gelu=-1) == mx.MX_ERR_INVALID_ARG
    assert call(bias=FAKE + 8 * MB + 4) == mx.MX_ERR_ALIGNMENT       # bias not 16-byte aligned
    assert call(bias=FAKE + 4 * MB + 256) == mx.MX_ERR_INVALID_ARG   # bias inside D
    # the NVFP4 form still needs its tensor scales
    ep = mx.mx_gemm_epilogue(None, 0.0, 1)
    assert lib.nvfp4_gemm_ex(FAKE, FAKE, FAKE, FAKE, None, None, FAKE, 128, 128, 256, 0, 1, 1,
                             ctypes.byref(ep), None, 0, None) == mx.MX_ERR_INVALID_ARG


def test_quantize_argument_validation(lib):
    q = lib.mx_quantize_bf16
    assert q(None, 4, 32, 32, 0, 0, FAKE, FAKE, None, None, 0, None) == mx.MX_ERR_INVALID_ARG
    assert q(FAKE, 4, 32, 16, 0, 0, FAKE, FAKE, None, None, 0, None) == mx.MX_ERR_INVALID_ARG
    assert q(FAKE, 4, 32, 32, 5, 0, FAKE, FAKE, None, None, 0, None) == mx.MX_ERR_INVALID_ARG
    assert q(FAKE, 4, 32, 32, 0, 9, FAKE, FAKE, None, None, 0, None) == mx.MX_ERR_INVALID_ARG
    assert q(FAKE, 4, 48, 48, 0, 0, FAKE, FAKE, None, None, 0, None) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert q(FAKE, 4, 32, 36, 0, 0, FAKE, FAKE, None, None, 0, None) == mx.MX_ERR_ALIGNMENT
    assert q(FAKE_ODD, 4, 32, 32, 0, 0, FAKE, FAKE, None, None, 0, None) == mx.MX_ERR_ALIGNMENT
    # MXFP4 takes no tensor scale; NVFP4 needs one and a workspace
    assert q(FAKE, 4, 32, 32, 0, 0, FAKE, FAKE, FAKE, None, 0, None) == mx.MX_ERR_INVALID_ARG
    assert q(FAKE, 4, 32, 32, 1, 0, FAKE, FAKE, None, None, 0, None) == mx.MX_ERR_INVALID_ARG
    assert q(FAKE, 4, 32, 32, 1, 0, FAKE, FAKE, FAKE, None, 0, None) == mx.MX_ERR_WORKSPACE


def test_quantize_sr_argument_validation(lib):
    q = lib.nvfp4_quantize_bf16_sr
    MB = 1 << 20

    def call(x=FAKE, rows=4, cols=32, ld=32, lay=0, c=FAKE + MB, s=FAKE + 2 * MB, ts=FAKE + 3 * MB,
             rounds=10, ws=FAKE + 4 * MB, wsb=1 << 16):
        return q(x, rows, cols, ld, lay, c, s, ts, 0x0123456789ABCDEF, rounds, ws, wsb, None)
    assert call(rounds=0) == mx.MX_ERR_INVALID_ARG
    assert call(rounds=mx.MX_PHILOX_MAX_ROUNDS + 1) == mx.MX_ERR_INVALID_ARG
    assert call(x=None) == mx.MX_ERR_INVALID_ARG
    assert call(ts=None) == mx.MX_ERR_INVALID_ARG                # NVFP4 needs the tensor scale
    assert call(lay=7) == mx.MX_ERR_INVALID_ARG
    assert call(cols=40, ld=40) == mx.MX_ERR_UNSUPPORTED_SHAPE    # cols % 16
    assert call(ld=36) == mx.MX_ERR_ALIGNMENT
    assert call(ts=FAKE + 3 * MB + 2) == mx.MX_ERR_ALIGNMENT
    assert call(ws=None) == mx.MX_ERR_WORKSPACE
    assert call(wsb=4) == mx.MX_ERR_WORKSPACE
    assert call(ws=FAKE_ODD) == mx.MX_ERR_ALIGNMENT


def test_nvfp4_quantize_2d_argument_validation(lib):
    MB = 1 << 20
    q = lib.nvfp4_quantize_bf16_2d
    ok = dict(x=FAKE, rows=64, cols=96, ld=96, lay=1, c=FAKE + MB, s=FAKE + 2 * MB,
              ct=FAKE + 3 * MB, st=FAKE + 4 * MB, ts=FAKE + 5 * MB, sr=1, rounds=10,
              ws=FAKE + 6 * MB, wsb=1 << 16)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return q(a["x"], a["rows"], a["cols"], a["ld"], a["lay"], a["c"], a["s"], a["ct"], a["st"],
                 a["ts"], a["sr"], 1234, a["rounds"], a["ws"], a["wsb"], None)
    assert call(x=None) == mx.MX_ERR_INVALID_ARG
    assert call(ct=None) == mx.MX_ERR_INVALID_ARG
    assert call(ts=None) == mx.MX_ERR_INVALID_ARG
    assert call(ld=64) == mx.MX_ERR_INVALID_ARG
    assert call(lay=3) == mx.MX_ERR_INVALID_ARG
    assert call(sr=2) == mx.MX_ERR_INVALID_ARG
    assert call(rounds=0) == mx.MX_ERR_INVALID_ARG
    assert call(rounds=17) == mx.MX_ERR_INVALID_ARG
    assert call(rows=40) == mx.MX_ERR_UNSUPPORTED_SHAPE           # rows % 16
    assert call(cols=88, ld=88) == mx.MX_ERR_UNSUPPORTED_SHAPE    # cols % 16
    assert call(st=FAKE_ODD) == mx.MX_ERR_ALIGNMENT
    assert call(ts=FAKE + 5 * MB + 2) == mx.MX_ERR_ALIGNMENT
    assert call(ld=100) == mx.MX_ERR_ALIGNMENT                    # ld % 8
    assert call(ws=None) == mx.MX_ERR_WORKSPACE
    assert call(wsb=8) == mx.MX_ERR_WORKSPACE
    assert call(ct=FAKE + MB + 64) == mx.MX_ERR_INVALID_ARG       # codes_t overlaps codes
    assert call(c=FAKE + 1024) == mx.MX_ERR_INVALID_ARG           # codes overlap the input
    assert call(ws=FAKE + 4 * MB) == mx.MX_ERR_INVALID_ARG        # workspace overlaps scales_t
    assert call(c=None) == mx.MX_ERR_INVALID_ARG                  # rowwise codes without scales
    # rounding to nearest ignores the round count
    assert call(sr=0, rounds=0, x=None) == mx.MX_ERR_INVALID_ARG


def _group(lib, tensors, fmt=0, layout=0, ws=None, wsb=0):
    arr = (mx.mx_quantize_tensor * max(1, len(tensors)))()
    for i, t in enumerate(tensors):
        arr[i] = mx.mx_quantize_tensor(*t)
    return lib.mx_quantize_bf16_group(arr, len(tensors), fmt, layout, ws, wsb, None)


def test_group_workspace_bytes(lib):
    per = mx.mx_quantize_workspace_bytes(1, 16, mx.MX_FMT_NVFP4)
    assert mx.mx_quantize_group_workspace_bytes(3, mx.MX_FMT_NVFP4) == 3 * per
    assert mx.mx_quantize_group_workspace_bytes(3, mx.MX_FMT_MXFP4) == 0
    assert mx.mx_quantize_group_workspace_bytes(0, mx.MX_FMT_NVFP4) == 0
    assert mx.mx_quantize_group_workspace_bytes(mx.MX_QUANTIZE_GROUP_MAX + 1, 1) == 0


def test_group_quantize_argument_validation(lib):
    MB = 1 << 20
    # (x, rows, cols, ld_x, codes, scales, tensor_scale): disjoint buffers 1 MiB apart
    t0 = (FAKE, 64, 256, 256, FAKE + 1 * MB, FAKE + 2 * MB, None)
    t1 = (FAKE + 3 * MB, 32, 512, 512, FAKE + 4 * MB, FAKE + 5 * MB, None)
    assert _group(lib, []) == mx.MX_ERR_INVALID_ARG                      # count 0
    assert _group(lib, [t0] * (mx.MX_QUANTIZE_GROUP_MAX + 1)) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_quantize_bf16_group(None, 1, 0, 0, None, 0, None) == mx.MX_ERR_INVALID_ARG
    # every tensor is checked as by mx_quantize_bf16
    assert _group(lib, [t0, t1[:1] + (32, 48, 48) + t1[4:]]) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert _group(lib, [t0, (FAKE_ODD,) + t1[1:]]) == mx.MX_ERR_ALIGNMENT
    assert _group(lib, [t0, t1[:6] + (FAKE + 6 * MB,)]) == mx.MX_ERR_INVALID_ARG  # MX tensor scale
    # outputs overlapping an input or another output are refused
    assert _group(lib, [t0, t1[:4] + (FAKE + 1 * MB,) + t1[5:]]) == mx.MX_ERR_INVALID_ARG
    assert _group(lib, [t0, t1[:4] + (FAKE + 16,) + t1[5:]]) == mx.MX_ERR_INVALID_ARG
    assert _group(lib, [t0[:5] + (FAKE + 1 * MB + 4096,) + t0[6:]]) == mx.MX_ERR_INVALID_ARG
    # NVFP4: tensor scales and a workspace of count x the per-tensor size
    n0 = t0[:6] + (FAKE + 6 * MB,)
    n1 = t1[:6] + (FAKE + 6 * MB + 64,)
    wsb = mx.mx_quantize_group_workspace_bytes(2, mx.MX_FMT_NVFP4)
    assert _group(lib, [n0, n1], fmt=1) == mx.MX_ERR_WORKSPACE
    assert _group(lib, [n0, n1], fmt=1, ws=FAKE + 7 * MB, wsb=wsb - 16) == mx.MX_ERR_WORKSPACE
    assert _group(lib, [n0, n0[:6] + (FAKE + 6 * MB,)], fmt=1, ws=FAKE + 7 * MB,
                  wsb=wsb) == mx.MX_ERR_INVALID_ARG                    # one shared tensor scale
    assert _group(lib, [n0, n1], fmt=1, ws=FAKE + 2 * MB, wsb=wsb) == mx.MX_ERR_INVALID_ARG


def test_quantize_2d_argument_validation(lib):
    MB = 1 << 20
    q = lib.mx_quantize_bf16_2d
    ok = dict(x=FAKE, rows=64, cols=96, ld=96, fmt=0, lay=1, c=FAKE + MB, s=FAKE + 2 * MB,
              ct=FAKE + 3 * MB, st=FAKE + 4 * MB)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return q(a["x"], a["rows"], a["cols"], a["ld"], a["fmt"], a["lay"], a["c"], a["s"], a["ct"],
                 a["st"], None)
    assert call(x=None) == mx.MX_ERR_INVALID_ARG
    assert call(ct=None) == mx.MX_ERR_INVALID_ARG
    assert call(ld=64) == mx.MX_ERR_INVALID_ARG
    assert call(lay=3) == mx.MX_ERR_INVALID_ARG
    assert call(fmt=1) == mx.MX_ERR_UNSUPPORTED_FEATURE          # NVFP4 not provided
    assert call(rows=48) == mx.MX_ERR_UNSUPPORTED_SHAPE           # rows % 32
    assert call(cols=80, ld=80) == mx.MX_ERR_UNSUPPORTED_SHAPE    # cols % 32
    assert call(st=FAKE_ODD) == mx.MX_ERR_ALIGNMENT
    assert call(ld=100) == mx.MX_ERR_ALIGNMENT                    # ld % 8
    assert call(ct=FAKE + MB + 64) == mx.MX_ERR_INVALID_ARG       # codes_t overlaps codes
    assert call(c=FAKE + 1024) == mx.MX_ERR_INVALID_ARG           # codes overlap the input
    assert call(c=None) == mx.MX_ERR_INVALID_ARG                  # rowwise codes without scales
    assert call(s=None) == mx.MX_ERR_INVALID_ARG


def test_relayout_and_selftest_validation(lib):
    assert lib.mx_scale_relayout(None, 4, 32, 0, FAKE, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_scale_relayout(FAKE, 4, 40, 0, FAKE, None) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert lib.mx_selftest_wait_timeout(0, None) == mx.MX_ERR_INVALID_ARG


def test_fp4_transpose_argument_validation(lib):
    t = lib.mx_fp4_transpose
    assert t(None, 64, 64, FAKE, None) == mx.MX_ERR_INVALID_ARG
    assert t(FAKE, 64, 64, None, None) == mx.MX_ERR_INVALID_ARG
    assert t(FAKE, 0, 64, FAKE + (1 << 20), None) == mx.MX_ERR_INVALID_ARG
    assert t(FAKE, 48, 64, FAKE + (1 << 20), None) == mx.MX_ERR_UNSUPPORTED_SHAPE   # rows % 32
    assert t(FAKE, 64, 80, FAKE + (1 << 20), None) == mx.MX_ERR_UNSUPPORTED_SHAPE   # cols % 32
    assert t(FAKE_ODD, 64, 64, FAKE + (1 << 20), None) == mx.MX_ERR_ALIGNMENT
    assert t(FAKE, 64, 64, FAKE + 1024, None) == mx.MX_ERR_INVALID_ARG             # overlap
    assert "overlaps" in mx.mx_last_error_string()
    assert t(FAKE, 64 * 65536, 64, FAKE + (1 << 36), None) == mx.MX_ERR_UNSUPPORTED_SHAPE


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="host without a GPU only")
def test_no_gpu_reports_unavailable(lib):
    assert mx.mx_available() is False
    # a well-formed call fails at the device check, not silently
    rc = _gemm(lib)
    assert rc in (mx.MX_ERR_CUDA, mx.MX_ERR_UNSUPPORTED_ARCH)


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library every call raises: there is no fallback path."""
    from block_scaled_fp4_bf16_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "libmxfp4.so"))
    with pytest.raises(RuntimeError, match="is missing"):
        _binding.mx_scale_bytes(128, 256, mx.MX_FMT_MXFP4, mx.MX_SCALE_TCGEN05)
    with pytest.raises(RuntimeError, match="is missing"):
        _binding.mx_available()


def test_static_workspace_rejects_oversized_partials_before_any_launch(lib):
    """Split-K partials beyond the fixed array (split_k * M * N * 4 bytes over
    MX_STATIC_WORKSPACE_BYTES) are refused with MX_ERR_WORKSPACE, and invalid
    arguments with the codes of mxfp4_gemm; no device is touched for either."""
    m, n, k = 128, 8192, 8192
    split = 8
    assert mx.mx_gemm_workspace_bytes(m, n, k, split) == split * m * n * 4
    assert split * m * n * 4 > mx.MX_STATIC_WORKSPACE_BYTES
    rc = lib.mxfp4_gemm_static_workspace(FAKE, FAKE, FAKE, FAKE, FAKE, m, n, k, 0, 0, split, None)
    assert rc == mx.MX_ERR_WORKSPACE
    rc = lib.mxfp4_gemm_static_workspace(None, FAKE, FAKE, FAKE, FAKE, 128, 128, 256, 0, 0, 1, None)
    assert rc == mx.MX_ERR_INVALID_ARG
    rc = lib.mxfp4_gemm_static_workspace(FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 128, 0, 0, 1, None)
    assert rc == mx.MX_ERR_UNSUPPORTED_SHAPE


def test_static_workspace_checks_arguments_before_the_partials_size(lib):
    """A call that is both invalid and oversized gets the code mxfp4_gemm gives
    for the invalid argument, not MX_ERR_WORKSPACE."""
    m, n, k, split = 128, 8192, 8192, 8
    assert split * m * n * 4 > mx.MX_STATIC_WORKSPACE_BYTES
    rc = lib.mxfp4_gemm_static_workspace(None, FAKE, FAKE, FAKE, FAKE, m, n, k, 0, 0, split, None)
    assert rc == mx.MX_ERR_INVALID_ARG
    rc = lib.mxfp4_gemm_static_workspace(FAKE, FAKE, FAKE, FAKE, FAKE, m, n, k, 1, 0, split, None)
    assert rc == mx.MX_ERR_UNSUPPORTED_FEATURE
    rc = lib.mxfp4_gemm_static_workspace(FAKE, FAKE, FAKE, FAKE, FAKE, m, n, k, 0, 5, split, None)
    assert rc == mx.MX_ERR_UNSUPPORTED_FEATURE
    rc = lib.mxfp4_gemm_static_workspace(FAKE, FAKE, FAKE, FAKE, FAKE, m, 8200, k, 0, 0, split,
                                         None)
    assert rc == mx.MX_ERR_UNSUPPORTED_SHAPE
    rc = lib.mxfp4_gemm_static_workspace(FAKE_ODD, FAKE, FAKE, FAKE, FAKE, m, n, k, 0, 0, split,
                                         None)
    assert rc == mx.MX_ERR_ALIGNMENT


def test_last_error_string_names_the_argument_and_constraint(lib):
    detail = lambda: lib.mx_last_error_string().decode()  # noqa: E731
    assert _gemm(lib, k=300) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert detail() == "mxfp4_gemm: K = 300 is not a multiple of 256"
    assert _gemm(lib, b=None) == mx.MX_ERR_INVALID_ARG
    assert detail() == "mxfp4_gemm: b_codes is null"
    assert _gemm(lib, n=40) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert detail() == "mxfp4_gemm: N = 40 is not a multiple of 32"
    assert _gemm(lib, layout=2) == mx.MX_ERR_UNSUPPORTED_FEATURE
    assert "layout 2" in detail()
    # quantize: the block of the format
    rc = lib.mx_quantize_bf16(FAKE, 4, 40, 40, mx.MX_FMT_NVFP4, 0, FAKE, FAKE, FAKE, FAKE,
                              4096, None)
    assert rc == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert detail() == "mx_quantize_bf16: cols = 40 is not a multiple of the NVFP4 block 16"
    # the NVFP4 amax workspace
    rc = lib.mx_quantize_bf16(FAKE, 4, 32, 32, mx.MX_FMT_NVFP4, 0, FAKE, FAKE, FAKE, FAKE, 16,
                              None)
    assert rc == mx.MX_ERR_WORKSPACE
    assert detail().startswith("mx_quantize_bf16: NVFP4 needs a workspace of 2048 bytes, got 16")
    # the static array's size, with the numbers
    rc = lib.mxfp4_gemm_static_workspace(FAKE, FAKE, FAKE, FAKE, FAKE, 128, 8192, 8192, 0, 0, 8,
                                         None)
    assert rc == mx.MX_ERR_WORKSPACE
    assert detail() == ("mxfp4_gemm_static_workspace: 8 splits of K need 33554432 bytes of "
                        "partial sums, more than the 16777216 bytes of the static array")
    # a group names the tensor
    t = (mx.mx_quantize_tensor * 2)()
    t[0].x, t[0].rows, t[0].cols, t[0].ld_x, t[0].codes, t[0].scales = FAKE, 4, 64, 64, FAKE, FAKE
    t[1].x, t[1].rows, t[1].cols, t[1].ld_x, t[1].codes, t[1].scales = FAKE, 4, 64, 32, FAKE, FAKE
    assert lib.mx_quantize_bf16_group(t, 2, mx.MX_FMT_MXFP4, 0, None, 0, None) == \
        mx.MX_ERR_INVALID_ARG
    assert detail().startswith("mx_quantize_bf16_group (tensor 1): rows, cols, ld_x = 4, 64, 32")


def test_last_error_string_is_per_thread_and_per_call(lib):
    import threading
    detail = lambda: lib.mx_last_error_string().decode()  # noqa: E731
    assert _gemm(lib, k=300) == mx.MX_ERR_UNSUPPORTED_SHAPE
    seen = {}

    def other():
        seen["before"] = detail()
        _gemm(lib, m=48)
        seen["after"] = detail()

    th = threading.Thread(target=other)
    th.start()
    th.join()
    assert seen["before"] == "no error recorded by the last call on this thread"
    assert seen["after"] == "mxfp4_gemm: M = 48 is not a multiple of 32"
    assert detail() == "mxfp4_gemm: K = 300 is not a multiple of 256"
    # the next call replaces it
    assert lib.mx_selftest_wait_timeout(0, None) == mx.MX_ERR_INVALID_ARG
    assert detail() == "mx_selftest_wait_timeout: timeout_ns = 0 (1 .. 1e10)"


def test_binding_errors_carry_the_detail(lib):
    with pytest.raises(mx.MXError, match="K = 300 is not a multiple of 256") as ei:
        mx.mxfp4_gemm(FAKE, FAKE, FAKE, FAKE, FAKE, 128, 128, 300, stream=0)
    assert ei.value.code == mx.MX_ERR_UNSUPPORTED_SHAPE


def test_calibrate_argument_validation(lib):
    flops = ctypes.c_double(0.0)
    units = ctypes.c_int(0)
    f, u = ctypes.byref(flops), ctypes.byref(units)
    assert lib.mx_calibrate_mma(3, 1, 16, None, 0, f, u, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_calibrate_mma(0, 2, 16, None, 0, f, u, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_calibrate_mma(0, 1, 0, None, 0, f, u, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_calibrate_mma(0, 1, mx.MX_CALIBRATE_MAX_STEPS + 1, None, 0, f, u, None) == \
        mx.MX_ERR_INVALID_ARG
    assert lib.mx_calibrate_mma(0, 1, 16, None, 0, None, u, None) == mx.MX_ERR_INVALID_ARG
    assert lib.mx_calibrate_mma(0, 1, 16, FAKE + 4, 152, f, u, None) == mx.MX_ERR_ALIGNMENT


def test_maximum_sizes_are_rejected_before_any_launch(lib):
    """The largest shapes the kernels' index arithmetic covers: beyond them
    every entry point answers MX_ERR_UNSUPPORTED_SHAPE (GEMM dimensions and
    quantize rows / cols below 2^31, fewer than 2^31 scale blocks, transpose
    rows below 64 * 65536), and the limit itself is accepted as far as the
    shape checks go (the fake pointers then fail the alignment check)."""
    big = 1 << 31
    assert _gemm(lib, m=big) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert _gemm(lib, n=big) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert _gemm(lib, k=big) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert _gemm(lib, m=big - 32, a=FAKE_ODD) == mx.MX_ERR_ALIGNMENT
    q = lib.mx_quantize_bf16
    # rows x (cols / 32) scale blocks reach 2^31 (cols = 2^16: 2^11 blocks a row)
    assert q(FAKE, 1 << 20, 1 << 16, 1 << 16, 0, 0, FAKE, FAKE, None, None, 0, None) == \
        mx.MX_ERR_UNSUPPORTED_SHAPE
    assert q(FAKE_ODD, (1 << 20) - 128, 1 << 16, 1 << 16, 0, 0, FAKE, FAKE, None, None, 0,
             None) == mx.MX_ERR_ALIGNMENT
    assert q(FAKE, big, 32, 32, 0, 0, FAKE, FAKE, None, None, 0, None) == \
        mx.MX_ERR_UNSUPPORTED_SHAPE
    t = lib.mx_fp4_transpose
    assert t(FAKE, 64 * 65536, 32, FAKE + (1 << 40), None) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert t(FAKE, 32, big, FAKE + (1 << 40), None) == mx.MX_ERR_UNSUPPORTED_SHAPE
    assert t(FAKE_ODD, 64 * 65535, 32, FAKE + (1 << 40), None) == mx.MX_ERR_ALIGNMENT
