"""GB300 (sm_103a) dense tensor-core GEMM  C = A . B^T  behind a C ABI."""
