"""fp64 CPU oracle of the DeepSeekMoE layer forward (test infrastructure only)."""
