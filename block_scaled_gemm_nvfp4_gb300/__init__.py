"""libnvfp4: NVFP4 quantisation and block-scaled FP4 GEMM for GB300 (sm_103a)."""
