"""CPU oracle (test infrastructure): see oracle/q8_oracle.py."""
