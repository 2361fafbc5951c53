"""Build the sm_103a CUDA library in-tree: block_scaled_fp4_bf16_gb300/_build/libmxfp4.so.

nvcc compiles each translation unit (in parallel) for sm_103a only and links
a shared library with the static CUDA runtime; the C ABI is include/mxfp4.h.
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
# MX_BOUNDS_CHECK=1 builds the bounds-checked library (-DMX_BOUNDS_CHECK: every
# plain global access of the kernels checked against its buffer, a test
# instrument) into its own folder; the binding then loads that one.
BOUNDS_CHECK = os.environ.get("MX_BOUNDS_CHECK") == "1"
OUT_DIR = os.path.join(PKG, "_build_bounds" if BOUNDS_CHECK else "_build")
LIB_PATH = os.path.join(OUT_DIR, "libmxfp4.so")
SOURCES = ["api.cu", "quantize.cu", "gemm.cu", "gemm_pair.cu", "gemm_swap.cu", "static_ws.cu",
           "calibrate.cu", "transpose.cu"]
HEADERS = ["mx_device.cuh", "mx_internal.h"]

ARCH_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH_FLAGS + [
    "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
    "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC,
]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _newest_input() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files += [os.path.join(INCLUDE, "mxfp4.h"), os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile (if stale) and return the path of libmxfp4.so."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= _newest_input():
        return LIB_PATH
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        objs.append(obj)
        flags = list(extra_flags) + (["-DMX_BOUNDS_CHECK"] if BOUNDS_CHECK else [])
        cmd = [nvcc()] + NVCC_FLAGS + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            print(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(" ".join(cmd))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    link = [nvcc()] + ARCH_FLAGS + ["-shared", "-o", tmp] + objs
    subprocess.run(link, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
