"""GB300-native FP4 block-scaled quantize-and-multiply (placeholder; the
binding to the CUDA library is added with the library)."""
