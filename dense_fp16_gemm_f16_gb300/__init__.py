"""GB300-native dense fp16 GEMM D = A·Bᵀ (binding added with the C-ABI)."""
