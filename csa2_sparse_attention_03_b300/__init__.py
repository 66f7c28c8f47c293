"""CSA2 decode hot path on B300 (placeholder; the binding is filled in below)."""
