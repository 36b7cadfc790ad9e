"""Float64 CPU oracle for the attention KL divergence (test infrastructure only)."""
