"""GB300-native batched speculative-sampling verification (placeholder; the
binding to the CUDA library is added with the kernels)."""
