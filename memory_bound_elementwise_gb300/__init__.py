"""GB300-native memory-bound elementwise operators (placeholder; binding added with the CUDA library)."""
