"""GB300-native deterministic top-k SwiGLU mixture-of-experts layer."""
