"""CPU oracle for the MoE / DeaMoE decode layer (test infrastructure only)."""
