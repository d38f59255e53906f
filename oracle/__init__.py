"""CPU oracle of the CTR sparse-embedding path (test infrastructure only)."""
