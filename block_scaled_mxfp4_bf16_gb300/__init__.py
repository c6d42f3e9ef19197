"""GB300-native block-scaled MXFP4 GEMM: C[M,N] (bf16) = MXFP4(A bf16) . MXFP4(B)^T."""
