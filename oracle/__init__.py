"""CPU oracle (test infrastructure only; see sparsp_oracle)."""
