"""GB300-native row-major FP32 GEMM (C = A x B) behind a small C ABI."""
