"""GB300-native Gated DeltaNet chunked-prefill forward (sm_103a CUDA behind a C ABI)."""
