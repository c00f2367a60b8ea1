"""fp64 CPU oracle of the gated delta rule (test infrastructure only; never imported by the
product path)."""
