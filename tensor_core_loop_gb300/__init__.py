"""GB300-native pipelined tensor-core GEMM (placeholder, binding added next)."""
