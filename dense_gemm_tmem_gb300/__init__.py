"""GB300-native dense GEMM library: C = A·B (+bias) on sm_103a."""
