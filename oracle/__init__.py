"""CPU oracle (test infrastructure only): see gq_oracle.c."""
