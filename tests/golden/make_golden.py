"""Write the oracle regression fixtures in this folder.

The block-scaled GEMM pages print no worked FP4 example, so the stored values
here are not the pages': they are written by this script, which calls only the
CPU oracle (and the seeded input generators), and they guard the oracle's
output against accidental change.  Re-run only when a change to the oracle's
arithmetic is justified by a passage of the pages (say which in the commit).

    python tests/golden/make_golden.py
"""
import json
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import numpy as np  # noqa: E402

import oracle  # noqa: E402
from block_scaled_fp4_bf16_gb300 import synth  # noqa: E402


def main():
    x = synth.bf16_normal(4, 64, 1.0, seed=0x601D)
    codes, scales = oracle.mx_quantize(x)
    nv_codes, nv_scales, s_t = oracle.nvfp4_quantize(x)
    a = synth.fp4_codes(32, 256, seed=0x601E)
    b = synth.fp4_codes(32, 256, seed=0x601F)
    sa = synth.scale_bytes(32, 8, 120, 134, seed=0x6020)
    sb = synth.scale_bytes(32, 8, 120, 134, seed=0x6021)
    d, s_abs = oracle.mx_gemm(a, sa, b, sb, 32, 32, 256, rows=[0, 5, 31], cols=[0, 17, 31])
    out = {
        "about": "oracle regression fixture written by make_golden.py (CPU oracle only)",
        "quantize_input_bf16_hex": [[f"{v:04x}" for v in row] for row in x.tolist()],
        "mx_codes_hex": [bytes(r).hex() for r in codes],
        "mx_scales": scales.tolist(),
        "nvfp4_codes_hex": [bytes(r).hex() for r in nv_codes],
        "nvfp4_scales": nv_scales.tolist(),
        "nvfp4_tensor_scale_hex": np.array([s_t], np.float32).view(np.uint32).tolist()[0],
        "gemm_seeds": [0x601E, 0x601F, 0x6020, 0x6021],
        "gemm_rows": [0, 5, 31], "gemm_cols": [0, 17, 31],
        "gemm_d": d.tolist(), "gemm_s_abs": s_abs.tolist(),
    }
    with open(os.path.join(HERE, "oracle_regression.json"), "w") as f:
        json.dump(out, f, indent=1)

    # stochastic rounding, the bidimensional NVFP4 quantize and the GEMM epilogue
    y = synth.bf16_normal(32, 64, 0.5, seed=0x6022)
    sr10, _, _ = oracle.nvfp4_quantize_sr(y, 0x0123456789ABCDEF, 10)
    sr7, _, _ = oracle.nvfp4_quantize_sr(y, 0x0123456789ABCDEF, 7)
    _, _, ct, st, _ = oracle.nvfp4_quantize_2d(y, seed=0x0123456789ABCDEF)
    draws = [oracle.philox4x32([j, r, d, 0], [0x89ABCDEF, 0x01234567], 10).tolist()
             for j, r, d in ((0, 0, 0), (3, 17, 0), (1, 2, 1))]
    bias = np.linspace(-1.0, 1.0, 3).astype(np.float32)
    c = np.arange(9, dtype=np.float64).reshape(3, 3) - 4.0
    epi = oracle.gemm_epilogue(d, bias=bias, gelu_on=True, beta=0.5, c=c)
    out2 = {
        "about": "oracle regression fixture written by make_golden.py (CPU oracle only)",
        "sr_input_seed": 0x6022, "sr_seed": 0x0123456789ABCDEF,
        "sr10_codes_hex": [bytes(r).hex() for r in sr10],
        "sr7_codes_hex": [bytes(r).hex() for r in sr7],
        "nv2d_sr_codes_t_hex": [bytes(r).hex() for r in ct],
        "nv2d_sr_scales_t": st.tolist(),
        "philox_draws": draws,
        "epilogue_bias": bias.tolist(), "epilogue_c": c.tolist(), "epilogue_beta": 0.5,
        "epilogue_gelu_d": epi.tolist(),
    }
    with open(os.path.join(HERE, "oracle_regression_sr_epilogue.json"), "w") as f:
        json.dump(out2, f, indent=1)


if __name__ == "__main__":
    main()
