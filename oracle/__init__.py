"""CPU oracle of the SPRINT decode step (test infrastructure only)."""
