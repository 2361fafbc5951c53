"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
(via the ctypes binding) on host inputs, and compare with the CPU oracle under
the tolerances of the block-scaled GEMM:

* quantize: codes, scales (and the NVFP4 tensor scale) byte-equal;
* FP32 out: |D - D_ref| <= 1e-5 * sum_k |a||b|;
* BF16 out: within 1 BF16 ulp of the correctly rounded D_ref, or (near
  cancellation, where the FP32 accumulation error exceeds a BF16 ulp of D)
  within the FP32 bound above; the count of the latter is reported.
"""
from __future__ import annotations

import numpy as np
import torch

import block_scaled_fp4_bf16_gb300 as mx
import oracle

FP32_REL_TOL = 1e-5

# Guard bands: every output a helper hands to the library sits between two
# GUARD_BYTES runs of GUARD_FILL bytes, checked after the call, so a write past
# either end of a buffer (a ragged tile, a padding row, a split-K partial)
# fails the test even when it lands in memory nothing else reads.  With
# compute-sanitizer unavailable, this and the bounds-checked build
# (-DMX_BOUNDS_CHECK) stand in for its memcheck.
GUARD_BYTES = 4096
GUARD_FILL = 0x5A


def guarded(n: int, dtype=torch.uint8, fill=None) -> torch.Tensor:
    """A contiguous device tensor of n elements with guard bands on both sides;
    the body is filled with `fill` (left at the guard pattern when None)."""
    esize = torch.empty((), dtype=dtype).element_size()
    nbytes = n * esize
    raw = torch.full((nbytes + 2 * GUARD_BYTES,), GUARD_FILL, dtype=torch.uint8, device="cuda")
    body = raw[GUARD_BYTES:GUARD_BYTES + nbytes].view(dtype)
    if fill is not None:
        body.fill_(fill)
    body._mx_guard = (raw, nbytes)
    return body


def check_guards(*tensors, what: str = ""):
    """Assert that no guard byte of the given guarded tensors changed."""
    for t in tensors:
        if t is None or not hasattr(t, "_mx_guard"):
            continue
        raw, nbytes = t._mx_guard
        for name, band in (("before", raw[:GUARD_BYTES]), ("after", raw[GUARD_BYTES + nbytes:])):
            bad = (band != GUARD_FILL).nonzero()
            if bad.numel():
                off = int(bad[0]) - (GUARD_BYTES if name == "before" else 0)
                raise AssertionError(f"{what}: {bad.numel()} byte(s) written {name} a buffer of "
                                     f"{nbytes} bytes (first at offset {off} from its "
                                     f"{'start' if name == 'before' else 'end'})")


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8)).cuda()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return torch.from_numpy(b.view(np.int16)).cuda().view(torch.bfloat16)


def gpu_quantize(x_bits: np.ndarray, fmt: int, layout: int, ld: int | None = None):
    """Quantize BF16 bits [rows, cols] on the GPU; returns host (codes, scales, s_t)."""
    rows, cols = x_bits.shape
    if ld is None or ld == cols:
        x = dev_bf16(x_bits)
        ld = cols
    else:
        padded = np.zeros((rows, ld), np.uint16)
        padded[:, :cols] = x_bits
        x = dev_bf16(padded)
    codes = guarded(rows * cols // 2, fill=0xAB)
    scales = guarded(mx.mx_scale_bytes(rows, cols, fmt, layout), fill=0xAB)
    ts = ws = None
    if fmt == mx.MX_FMT_NVFP4:
        ts = guarded(1, torch.float32, -1.0)
        ws = guarded(mx.mx_quantize_workspace_bytes(rows, cols, fmt))
    mx.mx_quantize_bf16(x, rows, cols, ld, fmt, layout, codes, scales, ts, ws)
    torch.cuda.synchronize()
    check_guards(codes, scales, ts, ws, what=f"quantize {rows}x{cols}")
    s_t = None if ts is None else np.float32(ts.item())
    return codes.cpu().numpy().reshape(rows, cols // 2), scales.cpu().numpy(), s_t


def gpu_quantize_sr(x_bits: np.ndarray, seed: int, rounds: int = 10, layout: int = 0,
                    ld: int | None = None):
    """NVFP4 quantize with stochastic rounding on the GPU (nvfp4_quantize_bf16_sr);
    returns host (codes, scales, s_t).  Outputs are pre-filled with 0xAB."""
    rows, cols = x_bits.shape
    ld = cols if ld is None else ld
    padded = np.zeros((rows, ld), np.uint16)
    padded[:, :cols] = x_bits
    x = dev_bf16(padded)
    fmt = mx.MX_FMT_NVFP4
    codes = guarded(rows * cols // 2, fill=0xAB)
    scales = guarded(mx.mx_scale_bytes(rows, cols, fmt, layout), fill=0xAB)
    ts = guarded(1, torch.float32, -1.0)
    ws = guarded(mx.mx_quantize_workspace_bytes(rows, cols, fmt))
    mx.nvfp4_quantize_bf16_sr(x, rows, cols, ld, layout, codes, scales, ts, seed, rounds, ws)
    torch.cuda.synchronize()
    check_guards(codes, scales, ts, ws, what=f"stochastic quantize {rows}x{cols}")
    return (codes.cpu().numpy().reshape(rows, cols // 2), scales.cpu().numpy(),
            np.float32(ts.item()))


def gpu_quantize_group(xs, fmt: int, layout: int, lds=None):
    """Quantize several BF16-bit arrays in one mx_quantize_bf16_group call;
    returns a list of host (codes, scales, s_t).  Outputs are pre-filled with
    0xAB so that any byte the kernel fails to write shows up."""
    lds = lds or [None] * len(xs)
    keep, tensors, outs = [], [], []
    for x_bits, ld in zip(xs, lds):
        rows, cols = x_bits.shape
        ld = cols if ld is None else ld
        padded = np.zeros((rows, ld), np.uint16)
        padded[:, :cols] = x_bits
        x = dev_bf16(padded)
        codes = guarded(rows * cols // 2, fill=0xAB)
        scales = guarded(mx.mx_scale_bytes(rows, cols, fmt, layout), fill=0xAB)
        ts = guarded(1, torch.float32, -1.0) if fmt == mx.MX_FMT_NVFP4 else None
        keep.append(x)
        tensors.append((x, rows, cols, ld, codes, scales, ts))
        outs.append((rows, cols, codes, scales, ts))
    wsb = mx.mx_quantize_group_workspace_bytes(len(xs), fmt)
    ws = guarded(wsb) if wsb else None
    mx.mx_quantize_bf16_group(tensors, fmt, layout, ws)
    torch.cuda.synchronize()
    for rows, cols, codes, scales, ts in outs:
        check_guards(codes, scales, ts, what=f"group quantize {rows}x{cols}")
    check_guards(ws, what="group quantize workspace")
    return [(codes.cpu().numpy().reshape(rows, cols // 2), scales.cpu().numpy(),
             None if ts is None else np.float32(ts.item())) for rows, cols, codes, scales, ts in outs]


def gpu_quantize_2d(x_bits: np.ndarray, layout: int, ld: int | None = None,
                    columnwise_only: bool = False):
    """Bidimensional MXFP4 quantize on the GPU; returns host (codes, scales,
    codes_t, scales_t), outputs pre-filled with 0xAB (codes and scales None
    when only the columnwise output is asked for)."""
    rows, cols = x_bits.shape
    ld = cols if ld is None else ld
    padded = np.zeros((rows, ld), np.uint16)
    padded[:, :cols] = x_bits
    x = dev_bf16(padded)
    fill = lambda n: guarded(n, fill=0xAB)  # noqa: E731
    fmt = mx.MX_FMT_MXFP4
    codes, codes_t = fill(rows * cols // 2), fill(rows * cols // 2)
    scales = fill(mx.mx_scale_bytes(rows, cols, fmt, layout))
    scales_t = fill(mx.mx_scale_bytes(cols, rows, fmt, layout))
    if columnwise_only:
        codes = scales = None
    mx.mx_quantize_bf16_2d(x, rows, cols, ld, fmt, layout, codes, scales, codes_t, scales_t)
    torch.cuda.synchronize()
    check_guards(codes, scales, codes_t, scales_t, what=f"bidimensional quantize {rows}x{cols}")
    return (None if codes is None else codes.cpu().numpy().reshape(rows, cols // 2),
            None if scales is None else scales.cpu().numpy(),
            codes_t.cpu().numpy().reshape(cols, rows // 2), scales_t.cpu().numpy())


def gpu_quantize_nv2d(x_bits: np.ndarray, layout: int, ld: int | None = None,
                      columnwise_only: bool = False, seed: int | None = None, rounds: int = 10):
    """Bidimensional NVFP4 quantize on the GPU (stochastic rounding when a seed
    is given); returns host (codes, scales, codes_t, scales_t, s_t), outputs
    pre-filled with 0xAB (codes and scales None for the columnwise output alone)."""
    rows, cols = x_bits.shape
    ld = cols if ld is None else ld
    padded = np.zeros((rows, ld), np.uint16)
    padded[:, :cols] = x_bits
    x = dev_bf16(padded)
    fill = lambda n: guarded(n, fill=0xAB)  # noqa: E731
    fmt = mx.MX_FMT_NVFP4
    codes, codes_t = fill(rows * cols // 2), fill(rows * cols // 2)
    scales = fill(mx.mx_scale_bytes(rows, cols, fmt, layout))
    scales_t = fill(mx.mx_scale_bytes(cols, rows, fmt, layout))
    ts = guarded(1, torch.float32, -1.0)
    ws = guarded(mx.mx_quantize_workspace_bytes(rows, cols, fmt))
    if columnwise_only:
        codes = scales = None
    mx.nvfp4_quantize_bf16_2d(x, rows, cols, ld, layout, codes, scales, codes_t, scales_t, ts,
                              0 if seed is None else 1, 0 if seed is None else seed, rounds, ws)
    torch.cuda.synchronize()
    check_guards(codes, scales, codes_t, scales_t, ts, ws,
                 what=f"bidimensional NVFP4 quantize {rows}x{cols}")
    return (None if codes is None else codes.cpu().numpy().reshape(rows, cols // 2),
            None if scales is None else scales.cpu().numpy(),
            codes_t.cpu().numpy().reshape(cols, rows // 2), scales_t.cpu().numpy(),
            np.float32(ts.item()))


def gpu_relayout(plain: np.ndarray, rows: int, cols: int, fmt: int) -> torch.Tensor:
    tiled = guarded(mx.mx_scale_bytes(rows, cols, fmt, mx.MX_SCALE_TCGEN05), fill=0xAB)
    mx.mx_scale_relayout(dev_u8(plain), rows, cols, fmt, tiled)
    torch.cuda.synchronize()
    check_guards(tiled, what=f"scale relayout {rows}x{cols}")
    return tiled


def gpu_gemm(fmt, a_codes, a_scales_tiled, b_codes, b_scales_tiled, m, n, k, out_fp32,
             split_k=0, a_ts=None, b_ts=None, prefill_nan=True):
    """Run the GEMM; operands may be host arrays or device tensors.  Returns host D
    (float32 array, or uint16 BF16 bits)."""
    def on_dev(a):
        return a if isinstance(a, torch.Tensor) else dev_u8(a)
    dt = torch.float32 if out_fp32 else torch.bfloat16
    body = guarded(m * n, dt, float("nan") if prefill_nan else 0.0)
    d = body.view(m, n)
    d._mx_guard = body._mx_guard
    wsb = mx.mx_gemm_workspace_bytes(m, n, k, split_k)
    ws = guarded(max(wsb, 16)) if wsb else None
    od = mx.MX_OUT_FP32 if out_fp32 else mx.MX_OUT_BF16
    if fmt == mx.MX_FMT_MXFP4:
        mx.mxfp4_gemm(on_dev(a_codes), on_dev(a_scales_tiled), on_dev(b_codes),
                      on_dev(b_scales_tiled), d, m, n, k, mx.MX_LAYOUT_TN, od, split_k, ws)
    else:
        ta = a_ts if isinstance(a_ts, torch.Tensor) else torch.tensor([a_ts], dtype=torch.float32,
                                                                      device="cuda")
        tb = b_ts if isinstance(b_ts, torch.Tensor) else torch.tensor([b_ts], dtype=torch.float32,
                                                                      device="cuda")
        mx.nvfp4_gemm(on_dev(a_codes), on_dev(a_scales_tiled), on_dev(b_codes),
                      on_dev(b_scales_tiled), ta, tb, d, m, n, k, mx.MX_LAYOUT_TN, od, split_k, ws)
    torch.cuda.synchronize()
    assert mx.mx_device_status() == mx.MX_OK
    check_guards(d, ws, what=f"GEMM {m}x{n}x{k} split {split_k}")
    if out_fp32:
        return d.cpu().numpy()
    return d.view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32).astype(np.float64)


def _bf16_ulp(bits: np.ndarray) -> np.ndarray:
    """Spacing of BF16 at each (finite) value: next-up minus value, in fp64."""
    mag = np.asarray(bits, np.uint16) & np.uint16(0x7FFF)
    v = bf16_bits_to_f64(mag)
    nxt = bf16_bits_to_f64(mag + np.uint16(1))
    return nxt - v


def check_fp32(d: np.ndarray, d_ref: np.ndarray, s_abs: np.ndarray, what: str = ""):
    d = np.asarray(d, np.float64)
    assert np.all(np.isfinite(d)), f"{what}: non-finite outputs"
    err = np.abs(d - d_ref)
    bound = FP32_REL_TOL * s_abs
    bad = err > bound
    if bad.any():
        i = np.argwhere(bad)[:5]
        raise AssertionError(
            f"{what}: {int(bad.sum())}/{bad.size} FP32 outputs out of tolerance; first "
            + ", ".join(f"{tuple(x)}: got {d[tuple(x)]!r} ref {d_ref[tuple(x)]!r} "
                        f"s_abs {s_abs[tuple(x)]!r}" for x in i))
    return float((err / np.maximum(s_abs, 1e-300)).max())


def check_bf16(d_bits: np.ndarray, d_ref: np.ndarray, s_abs: np.ndarray, what: str = ""):
    d_bits = np.asarray(d_bits, np.uint16)
    d = bf16_bits_to_f64(d_bits)
    assert np.all(np.isfinite(d)), f"{what}: non-finite outputs"
    ref_bits = oracle.round_bf16(d_ref)
    ref = bf16_bits_to_f64(ref_bits)
    ulp = _bf16_ulp(ref_bits)
    within_ulp = np.abs(d - ref) <= ulp
    within_fp32 = np.abs(d - d_ref) <= FP32_REL_TOL * s_abs
    ok = within_ulp | within_fp32
    if not ok.all():
        i = np.argwhere(~ok)[:5]
        raise AssertionError(
            f"{what}: {int((~ok).sum())}/{ok.size} BF16 outputs out of tolerance; first "
            + ", ".join(f"{tuple(x)}: got {d[tuple(x)]!r} ref {d_ref[tuple(x)]!r}" for x in i))
    return {"exact": int((d_bits == ref_bits).sum()), "within_1ulp": int(within_ulp.sum()),
            "only_fp32_rule": int((~within_ulp & within_fp32).sum()), "total": int(ok.size)}


def sample_indices(n: int, count: int, tile: int, seed: int) -> np.ndarray:
    """Deterministic sample of indices covering the first and last tile and random interior."""
    rng = np.random.default_rng(seed)
    idx = set(range(min(n, 8))) | set(range(max(0, n - 8), n))
    idx |= {min(n - 1, t) for t in (tile - 1, tile, 2 * tile - 1)}
    if n > 0:
        idx |= set(rng.integers(0, n, size=count).tolist())
    return np.array(sorted(idx), dtype=np.int64)
