"""CPU oracle for the quantized decode GEMM (test infrastructure only)."""
