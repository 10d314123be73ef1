"""GB300-native virtual-rank sum all-reduce (binding is added with the CUDA library)."""
