"""Float64 CPU oracle (test infrastructure only; see spec_oracle.py)."""
