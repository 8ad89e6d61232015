"""CPU oracle for the CRISP sparse-prefill path: test infrastructure only.

Imported only by tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg.
"""
