"""CPU oracle for the MoE expert-FFN layer (test infrastructure only; see oracle.py)."""
