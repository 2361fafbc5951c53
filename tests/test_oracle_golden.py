"""The oracle still reproduces its stored regression fixture."""
import json
import os

import numpy as np

from block_scaled_fp4_bf16_gb300 import synth

HERE = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def test_oracle_regression_fixture(oracle):
    g = json.load(open(os.path.join(HERE, "oracle_regression.json")))
    x = np.array([[int(v, 16) for v in row] for row in g["quantize_input_bf16_hex"]], np.uint16)
    assert np.array_equal(x, synth.bf16_normal(4, 64, 1.0, seed=0x601D))
    codes, scales = oracle.mx_quantize(x)
    assert [bytes(r).hex() for r in codes] == g["mx_codes_hex"]
    assert scales.tolist() == g["mx_scales"]
    nc, ns, s_t = oracle.nvfp4_quantize(x)
    assert [bytes(r).hex() for r in nc] == g["nvfp4_codes_hex"]
    assert ns.tolist() == g["nvfp4_scales"]
    assert np.array([s_t], np.float32).view(np.uint32)[0] == g["nvfp4_tensor_scale_hex"]
    sa_, sb_, sc_, sd_ = g["gemm_seeds"]
    a = synth.fp4_codes(32, 256, seed=sa_)
    b = synth.fp4_codes(32, 256, seed=sb_)
    sa = synth.scale_bytes(32, 8, 120, 134, seed=sc_)
    sb = synth.scale_bytes(32, 8, 120, 134, seed=sd_)
    d, s_abs = oracle.mx_gemm(a, sa, b, sb, 32, 32, 256, rows=g["gemm_rows"], cols=g["gemm_cols"])
    assert d.tolist() == g["gemm_d"]
    assert s_abs.tolist() == g["gemm_s_abs"]
