"""CPU oracle for the low-bit linear layer (test infrastructure; see oracle.py)."""
