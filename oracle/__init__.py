"""fp64 CPU oracle of the k-quant routed-MoE layer (test infrastructure only)."""
