"""fp64 CPU oracle for the packed double-binary matmul (test infrastructure only)."""
