"""CPU oracle (test infrastructure only; see lb_oracle)."""
