"""Plain CPU oracle of the MoE-layer forward (test infrastructure only)."""
