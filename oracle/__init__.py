"""CPU oracle for the block-quantized KV cache (test infrastructure only)."""
