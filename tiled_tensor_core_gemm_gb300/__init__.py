"""GB300-native dense GEMM: C = A.B over row-major operands, FP32 output."""
