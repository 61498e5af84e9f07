"""Plain fp64 CPU oracle for the sharded Muon step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product path never does.
"""
