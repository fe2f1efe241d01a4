"""GB300-native persistent / SM-constrained / Stream-K addmm GEMM (bf16 and MXFP4)."""
