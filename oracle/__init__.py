"""CPU oracle of the MoE block forward (test infrastructure only; see oracle.py)."""
