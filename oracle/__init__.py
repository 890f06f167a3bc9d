"""CPU oracle of the XPress Jacobi refinement pass (test infrastructure only)."""
