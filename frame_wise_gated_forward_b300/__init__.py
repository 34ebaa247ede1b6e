"""B300-native frame-wise Gated DeltaNet forward (sm_103a CUDA behind a C ABI)."""
