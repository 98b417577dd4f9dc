"""GB300-native chunked (ring) attention forward: C-ABI CUDA library + binding."""
