"""CPU oracle of the OScaR INT2 KV-cache hot path (test infrastructure only)."""
