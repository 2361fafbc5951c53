"""Seeded synthetic inputs for the block-scaled FP4 GEMM workloads.

This module holds input generation only (no quantization, decoding or GEMM
arithmetic), so that the CPU oracle and the CUDA path can be fed identical
bytes.  Everything is numpy on the host and deterministic for a given seed:

* BF16 matrices ~ N(0, sigma): numpy's counter-based Philox generator draws
  binary32 normals, scaled by sigma in binary32 and rounded to BF16
  (round-to-nearest-even on the bit pattern).
* FP4 code bytes: uniform over 0..255, so every one of the 16 E2M1 codes
  (including -0, code 8) appears in both nibbles.
* Scale bytes: uniform integers in [lo, hi].

Shapes follow the workloads of the block-scaled GEMM pages: activations
A [M, K] and weights W [N, K], both K-contiguous (TN).
"""
from __future__ import annotations

import numpy as np

# Base seed of every workload; workload i uses BASE_SEED + i.
BASE_SEED = 0x5EED


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.Philox(int(seed)))


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """binary32 -> BF16 bit patterns, round-to-nearest-even (finite inputs)."""
    u = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    bias = ((u >> np.uint32(16)) & np.uint32(1)) + np.uint32(0x7FFF)
    return ((u + bias) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_normal(rows: int, cols: int, sigma: float, seed: int,
                chunk: int = 1 << 24) -> np.ndarray:
    """BF16 bits [rows, cols] drawn from N(0, sigma^2)."""
    rng = _rng(seed)
    n = rows * cols
    out = np.empty(n, dtype=np.uint16)
    s = np.float32(sigma)
    for start in range(0, n, chunk):
        cnt = min(chunk, n - start)
        f = rng.standard_normal(cnt, dtype=np.float32)
        f *= s
        out[start:start + cnt] = f32_to_bf16_bits(f)
    return out.reshape(rows, cols)


def fp4_codes(rows: int, k: int, seed: int) -> np.ndarray:
    """Packed FP4 code bytes [rows, k/2], every byte value equally likely."""
    return _rng(seed).integers(0, 256, size=(rows, k // 2), dtype=np.uint8)


def scale_bytes(rows: int, kb: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Scale bytes [rows, kb] uniform over the integers lo..hi."""
    return _rng(seed).integers(lo, hi + 1, size=(rows, kb), dtype=np.uint8)


# --------------------------------------------------------------------------
# The workloads of the block-scaled GEMM and its quantizers (sizes and
# distributions).
# --------------------------------------------------------------------------

WORKLOADS = {
    # MXFP4 GEMM on seed-generated codes and scales, FP32 out.
    "mxfp4_128x128x256": dict(kind="codes", fmt="mxfp4", m=128, n=128, k=256,
                              scale_lo=120, scale_hi=134, out="fp32", split_k=1),
    # BF16 activations and weights quantized to MXFP4, BF16 out.
    "quant_gemm_2048x4096x4096": dict(kind="bf16", fmt="mxfp4", m=2048, n=4096, k=4096,
                                      sigma_a=1.0, sigma_b=0.02, out="bf16", split_k=1),
    # The same step with the GEMM epilogue D = GELU(A W^T + bias), FP32 bias [N].
    "quant_gemm_bias_gelu_2048x4096x4096": dict(kind="bf16", fmt="mxfp4", m=2048, n=4096, k=4096,
                                                sigma_a=1.0, sigma_b=0.02, out="bf16", split_k=1,
                                                bias=True, sigma_bias=1.0, gelu=True),
    # LLM MLP up-projection, compute bound.
    "mlp_up_16384x28672x8192": dict(kind="bf16", fmt="mxfp4", m=16384, n=28672, k=8192,
                                    sigma_a=1.0, sigma_b=0.015, out="bf16", split_k=1),
    # Decode-shaped skinny GEMM, split-K, HBM bound on B.
    "skinny_32x8192x8192": dict(kind="codes", fmt="mxfp4", m=32, n=8192, k=8192,
                                scale_lo=122, scale_hi=130, out="bf16", split_k=0),
    # NVFP4 variant, FP32 out.
    "nvfp4_4096x4096x4096": dict(kind="bf16", fmt="nvfp4", m=4096, n=4096, k=4096,
                                 sigma_a=1.0, sigma_b=1.0, out="fp32", split_k=1),
    # Bidimensional MXFP4 quantize (rowwise + columnwise) of the MLP weight
    # 28672 x 8192: no GEMM (n = 0), HBM bound.
    "quant2d_28672x8192": dict(kind="quant2d", fmt="mxfp4", m=28672, n=0, k=8192,
                               sigma_a=0.015, out="codes", split_k=1),
    # NVFP4 quantize with stochastic rounding (Philox4x32-10 per block) of a
    # 16384 x 8192 gradient-like tensor: no GEMM (n = 0), HBM bound.
    "nvfp4_sr_16384x8192": dict(kind="quant_sr", fmt="nvfp4", m=16384, n=0, k=8192,
                                sigma_a=1e-3, out="codes", split_k=1),
    # Bidimensional NVFP4 quantize with stochastic rounding (rowwise and
    # columnwise outputs) of the same tensor: no GEMM, HBM bound.
    "nvfp4_quant2d_sr_16384x8192": dict(kind="quant2d", fmt="nvfp4", sr=True, m=16384, n=0,
                                        k=8192, sigma_a=1e-3, out="codes", split_k=1),
    # The same bidimensional NVFP4 quantize with rounding to nearest.
    "nvfp4_quant2d_16384x8192": dict(kind="quant2d", fmt="nvfp4", sr=False, m=16384, n=0,
                                     k=8192, sigma_a=1e-3, out="codes", split_k=1),
    # The NVFP4 workload's shape and inputs in MXFP4: the two formats' GEMM
    # kernels side by side.
    "mxfp4_4096x4096x4096": dict(kind="bf16", fmt="mxfp4", m=4096, n=4096, k=4096,
                                 sigma_a=1.0, sigma_b=1.0, out="fp32", split_k=1),
    # FP4 codes of the MLP weight stored K x N (N contiguous, the NN / TN
    # operand order of a layer's weight) transposed to N x K for the GEMM:
    # no GEMM (n = 0), HBM bound.  Codes uniform over all 16 values.
    "fp4_transpose_8192x28672": dict(kind="transpose", fmt="mxfp4", m=8192, n=0, k=28672,
                                     out="codes", split_k=1),
    # Decode step of the MLP up-projection: 32 tokens x the 28672 x 8192
    # weight, HBM bound on the weight (more 128-row slices than SMs).
    "decode_mlp_up_32x28672x8192": dict(kind="codes", fmt="mxfp4", m=32, n=28672, k=8192,
                                        scale_lo=122, scale_hi=130, out="bf16", split_k=0),
}
WORKLOAD_ORDER = list(WORKLOADS)


def workload_seed(name: str) -> int:
    return BASE_SEED + WORKLOAD_ORDER.index(name)


def workload_inputs(name: str, m: int | None = None, n: int | None = None,
                    k: int | None = None) -> dict:
    """Host inputs of a workload (optionally at other sizes with the same recipe).

    kind == "bf16": {"a": BF16 bits [m, k], "b": BF16 bits [n, k]} (+ "bias": FP32 [n]
                    for a workload with a bias)
    kind == "codes": {"a_codes", "a_scales", "b_codes", "b_scales"} (plain scales)
    kind == "quant2d" or "quant_sr": {"a": BF16 bits [m, k]}
    kind == "transpose": {"a_codes": FP4 codes [m, k / 2]}
    """
    w = WORKLOADS[name]
    m = w["m"] if m is None else m
    n = w["n"] if n is None else n
    k = w["k"] if k is None else k
    seed = workload_seed(name) * 16
    if w["kind"] == "bf16":
        out = {"a": bf16_normal(m, k, w["sigma_a"], seed + 1),
               "b": bf16_normal(n, k, w["sigma_b"], seed + 2)}
        if w.get("bias"):
            rng = np.random.Generator(np.random.Philox(seed + 3))
            out["bias"] = (rng.standard_normal(n, dtype=np.float32) * np.float32(w["sigma_bias"]))
        return out
    if w["kind"] in ("quant2d", "quant_sr"):
        return {"a": bf16_normal(m, k, w["sigma_a"], seed + 1)}
    if w["kind"] == "transpose":
        return {"a_codes": fp4_codes(m, k, seed + 1)}
    kb = k // 32
    return {"a_codes": fp4_codes(m, k, seed + 1),
            "a_scales": scale_bytes(m, kb, w["scale_lo"], w["scale_hi"], seed + 2),
            "b_codes": fp4_codes(n, k, seed + 3),
            "b_scales": scale_bytes(n, kb, w["scale_lo"], w["scale_hi"], seed + 4)}
