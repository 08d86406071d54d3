"""fp64 CPU oracle of the chunked LM-head cross-entropy (test infrastructure only)."""
