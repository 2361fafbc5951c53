"""GB300 (sm_103a) MXFP4 / NVFP4 block-scaled GEMM and BF16 quantizer."""
