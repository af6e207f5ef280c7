"""W4A16 skinny GEMM for GB300 (sm_103a): Python binding of the C-ABI library."""
