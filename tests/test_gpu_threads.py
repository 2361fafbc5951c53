"""The C ABI is stateless and thread-safe: host threads may call it at once on
their own streams, also for the first calls of a process, when each kernel's
launch set-up (shared-memory limit, occupancy) is made and recorded.  A fresh
process starts eight threads together (a barrier), each making the first call
of a different kind on its own stream: the grouped MXFP4 quantize, the pair
GEMM, the swapped GEMM with a cluster split, the single-CTA GEMM with a
workspace split, the NVFP4 quantize and GEMM, the bidimensional quantize and
the transpose.  Every result must equal the same call made again afterwards on
one thread, byte for byte, and the device status word must stay clean."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r'''
import sys, threading
import numpy as np
import torch
import block_scaled_fp4_bf16_gb300 as mx
from block_scaled_fp4_bf16_gb300 import synth

MX, NV, T = mx.MX_FMT_MXFP4, mx.MX_FMT_NVFP4, mx.MX_SCALE_TCGEN05
torch.cuda.set_device(0)
dev = "cuda"

def bf16(r, c, sigma, seed):
    b = synth.bf16_normal(r, c, sigma, seed=seed).view(np.int16)
    return torch.from_numpy(b).to(dev).view(torch.bfloat16)

def u8(n):
    return torch.empty(n, dtype=torch.uint8, device=dev)

def codes_of(r, c, seed):
    return torch.from_numpy(synth.fp4_codes(r, c, seed)).to(dev)

def scales_of(r, c, seed):
    plain = torch.from_numpy(synth.scale_bytes(r, c // 32, 120, 134, seed)).to(dev)
    t = u8(mx.mx_scale_bytes(r, c, MX, T))
    mx.mx_scale_relayout(plain, r, c, MX, t)
    return t

# inputs, made before the threads start
xa, xw = bf16(256, 512, 1.0, 1), bf16(384, 512, 0.05, 2)
gemm_in = {}
for name, (m, n, k) in {"pair": (512, 768, 1024), "swap": (32, 1024, 2048),
                        "single": (96, 512, 1024)}.items():
    gemm_in[name] = (codes_of(m, k, 10 + m), scales_of(m, k, 20 + m), codes_of(n, k, 30 + n),
                     scales_of(n, k, 40 + n), m, n, k)
torch.cuda.synchronize()

def job(kind, stream):
    """One call of `kind` on `stream`; returns its outputs (device tensors)."""
    with torch.cuda.stream(stream):
        if kind == "group":
            out = [u8(256 * 256), u8(mx.mx_scale_bytes(256, 512, MX, T)),
                   u8(384 * 256), u8(mx.mx_scale_bytes(384, 512, MX, T))]
            mx.mx_quantize_bf16_group([(xa, 256, 512, 512, out[0], out[1], None),
                                       (xw, 384, 512, 512, out[2], out[3], None)], MX, T,
                                      u8(16), stream=stream)
        elif kind in ("pair", "swap", "single"):
            a, sa, b, sb, m, n, k = gemm_in[kind]
            d = torch.empty((m, n), dtype=torch.bfloat16, device=dev)
            split = 2 if kind == "single" else 0
            wsb = mx.mx_gemm_workspace_bytes(m, n, k, split)
            ws = u8(max(16, wsb))
            mx.mxfp4_gemm(a, sa, b, sb, d, m, n, k, split_k=split, workspace=ws,
                          workspace_bytes=wsb, stream=stream)
            out = [d.view(torch.int16)]
        elif kind == "nvfp4":
            ca, sa_, ta = u8(256 * 256), u8(mx.mx_scale_bytes(256, 512, NV, T)), \
                torch.empty(1, dtype=torch.float32, device=dev)
            cb, sb_, tb = u8(384 * 256), u8(mx.mx_scale_bytes(384, 512, NV, T)), \
                torch.empty(1, dtype=torch.float32, device=dev)
            mx.mx_quantize_bf16(xa, 256, 512, 512, NV, T, ca, sa_, ta,
                                u8(mx.mx_quantize_workspace_bytes(256, 512, NV)), stream=stream)
            mx.mx_quantize_bf16(xw, 384, 512, 512, NV, T, cb, sb_, tb,
                                u8(mx.mx_quantize_workspace_bytes(384, 512, NV)), stream=stream)
            d = torch.empty((256, 384), dtype=torch.float32, device=dev)
            mx.nvfp4_gemm(ca, sa_, cb, sb_, ta, tb, d, 256, 384, 512, stream=stream)
            out = [ca, sa_, cb, sb_, ta.view(torch.int32), d.view(torch.int32)]
        elif kind == "q2d":
            out = [u8(256 * 256), u8(mx.mx_scale_bytes(256, 512, MX, T)), u8(256 * 256),
                   u8(mx.mx_scale_bytes(512, 256, MX, T))]
            mx.mx_quantize_bf16_2d(xa, 256, 512, 512, MX, T, *out, stream=stream)
        elif kind == "transpose":
            a = gemm_in["pair"][0]
            out = [u8(512 * 1024 // 2)]
            mx.mx_fp4_transpose(a, 512, 1024, out[0], stream=stream)
    stream.synchronize()
    return [t.cpu().numpy().copy() for t in out]

KINDS = ["group", "pair", "swap", "single", "nvfp4", "q2d", "transpose", "pair"]
results, errors = [None] * len(KINDS), []
start = threading.Barrier(len(KINDS))

def worker(i, kind):
    try:
        stream = torch.cuda.Stream()
        start.wait()
        results[i] = job(kind, stream)
    except BaseException as e:
        errors.append(f"{kind}: {e!r}")

threads = [threading.Thread(target=worker, args=(i, k)) for i, k in enumerate(KINDS)]
for t in threads:
    t.start()
for t in threads:
    t.join()
assert not errors, errors
for i, kind in enumerate(KINDS):
    again = job(kind, torch.cuda.Stream())
    assert len(again) == len(results[i])
    for x, y in zip(results[i], again):
        assert np.array_equal(x, y), f"{kind}: the concurrent call differs from the sequential one"
assert mx.mx_device_status() == 0
print("threads ok")
'''


def test_concurrent_first_calls_from_threads():
    env = dict(os.environ)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True,
                       text=True, timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
