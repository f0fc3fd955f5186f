"""CPU oracle (test infrastructure only): see csa2_oracle.py."""
