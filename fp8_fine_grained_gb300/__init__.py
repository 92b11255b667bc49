"""Fine-grained FP8 quantisation and block-scaled FP8 GEMM for GB300 (sm_103a)."""
