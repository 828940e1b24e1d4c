"""libhgemm: half-precision tensor-core GEMM for GB300 (sm_103a)."""
