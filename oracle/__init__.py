"""CPU oracle (test infrastructure only; see dustin_oracle.py)."""
