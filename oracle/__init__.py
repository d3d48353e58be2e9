"""CPU oracle of the decode step (test infrastructure; see oracle.py)."""
