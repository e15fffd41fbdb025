"""CPU oracle for the W12 verify path (test infrastructure only; see w12_oracle)."""
