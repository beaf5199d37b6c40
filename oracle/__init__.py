"""fp64 CPU oracle of the quantised routed-MoE layer (test infrastructure only)."""
