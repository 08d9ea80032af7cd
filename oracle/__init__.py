"""CPU oracle for absorbed MLA (test infrastructure only; see mla_oracle)."""
