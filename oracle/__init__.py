"""CPU oracle for WISE paged decode attention (test infrastructure only)."""
