"""CPU oracle for the hybrid-batch layer (test infrastructure only)."""
