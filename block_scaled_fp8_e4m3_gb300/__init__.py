"""Block-scaled FP8 (E4M3) quantization, GEMM and weight sync for GB300."""
