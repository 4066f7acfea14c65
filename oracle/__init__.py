"""CPU oracle (test infrastructure only; see e0_oracle's module docstring)."""
