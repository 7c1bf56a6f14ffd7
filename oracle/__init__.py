"""CPU oracle for the Mamba-3 scan: test infrastructure only (see oracle.py)."""
