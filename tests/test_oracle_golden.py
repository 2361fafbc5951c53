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


def test_oracle_regression_fixture_sr_and_epilogue(oracle):
    g = json.load(open(os.path.join(HERE, "oracle_regression_sr_epilogue.json")))
    y = synth.bf16_normal(32, 64, 0.5, seed=g["sr_input_seed"])
    seed = g["sr_seed"]
    c10, _, _ = oracle.nvfp4_quantize_sr(y, seed, 10)
    c7, _, _ = oracle.nvfp4_quantize_sr(y, seed, 7)
    assert [bytes(r).hex() for r in c10] == g["sr10_codes_hex"]
    assert [bytes(r).hex() for r in c7] == g["sr7_codes_hex"]
    _, _, ct, st, _ = oracle.nvfp4_quantize_2d(y, seed=seed)
    assert [bytes(r).hex() for r in ct] == g["nv2d_sr_codes_t_hex"]
    assert st.tolist() == g["nv2d_sr_scales_t"]
    draws = [oracle.philox4x32([j, r, d, 0], [0x89ABCDEF, 0x01234567], 10).tolist()
             for j, r, d in ((0, 0, 0), (3, 17, 0), (1, 2, 1))]
    assert draws == g["philox_draws"]
    gg = json.load(open(os.path.join(HERE, "oracle_regression.json")))
    a = synth.fp4_codes(32, 256, seed=gg["gemm_seeds"][0])
    b = synth.fp4_codes(32, 256, seed=gg["gemm_seeds"][1])
    sa = synth.scale_bytes(32, 8, 120, 134, seed=gg["gemm_seeds"][2])
    sb = synth.scale_bytes(32, 8, 120, 134, seed=gg["gemm_seeds"][3])
    d, _ = oracle.mx_gemm(a, sa, b, sb, 32, 32, 256, rows=gg["gemm_rows"], cols=gg["gemm_cols"])
    epi = oracle.gemm_epilogue(d, bias=np.float32(g["epilogue_bias"]), gelu_on=True,
                               beta=g["epilogue_beta"], c=np.array(g["epilogue_c"]))
    assert epi.tolist() == g["epilogue_gelu_d"]
