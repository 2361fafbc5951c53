"""The CPU oracle samples that bench.py times (cpu_baseline and the reference
arm): a GEMM step is cut into an output block plus the matching share of the
quantize work, so that a tiny sample is valid and cheap and a run of many
steps stays bounded."""
import math
import os
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from block_scaled_fp4_bf16_gb300 import synth  # noqa: E402


@pytest.fixture(scope="module")
def skinny():
    name = "skinny_32x8192x8192"
    host = synth.workload_inputs(name)
    return name, host, bench.oracle_prepare(name, host)


def test_smallest_gemm_sample_is_a_few_outputs(skinny):
    """The floor the reference arm may ask for (one output's share) runs a
    block of at least one row: here 1 x 16 outputs of 32 x 8192, at once."""
    name, host, prepared = skinny
    _, m, n, _ = bench.workload_shape(name)
    t0 = time.perf_counter()
    t, f = bench.oracle_step_sample(name, host, 1.0 / (m * n), prepared)
    assert f * m * n == 16
    assert time.perf_counter() - t0 < 5.0 and t > 0.0


def test_gemm_sample_is_a_block_of_the_output(skinny):
    name, host, prepared = skinny
    _, m, n, _ = bench.workload_shape(name)
    frac = 1.0 / 64
    _, f = bench.oracle_step_sample(name, host, frac, prepared)
    g = math.sqrt(frac)
    assert f == round(m * g) * round(n * g) / (m * n)
    assert bench.gemm_block(f, m, n) == f"a {round(m * g)} x {round(n * g)} block of the 32 x 8192 output"


def test_quantize_sample_takes_whole_rows():
    name = "nvfp4_sr_16384x8192"
    _, m, _, _ = bench.workload_shape(name)
    host = {"a": synth.bf16_normal(64, 8192, 1e-3, seed=5)}
    _, f = bench.oracle_step_sample(name, host, 48 / m, None)
    assert f == 48 / m
