"""CPU fp64 oracle for fused linear cross-entropy (test infrastructure only)."""
