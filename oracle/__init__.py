"""CPU oracle for the MX hot path (test infrastructure; see mx_oracle)."""
