"""CPU oracle for the block-scaled FP8 GEMM (test infrastructure only; see oracle.cpp)."""
