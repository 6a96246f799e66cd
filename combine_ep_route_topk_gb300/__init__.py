"""GB300-native MoE expert-parallel route / layout / dispatch / combine."""
