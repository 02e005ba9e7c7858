"""GB300-native GGUF block-quantized matmul (placeholder; binding added below)."""
