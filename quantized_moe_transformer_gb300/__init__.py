"""GB300-native k-quant routed-MoE layer: C-ABI CUDA library plus a thin binding."""
