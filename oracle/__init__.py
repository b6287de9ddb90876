"""fp64 CPU oracle (test infrastructure only; see cross_attention.py)."""
