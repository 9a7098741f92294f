"""fp64 CPU oracle for block-sparse attention forward.  Test infrastructure only:
imported by tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg, never by
the product package."""
