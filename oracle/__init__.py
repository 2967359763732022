"""CPU oracle of the routed MoE forward (test infrastructure only)."""
