"""GB300-native lossless compression of float model tensors (placeholder)."""
