"""CSA2 oracle package (test infrastructure only; see oracle.oracle)."""
