"""fp64 CPU oracle for attention forward/backward: test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the library never does.
"""
