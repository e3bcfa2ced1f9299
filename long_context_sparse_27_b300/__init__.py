"""CSA2 global-attention step on B300 (placeholder; the binding lands with the library)."""
