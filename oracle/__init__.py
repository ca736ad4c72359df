"""fp64 CPU oracle (test infrastructure): see spec_verify_oracle.py and exact.py."""
