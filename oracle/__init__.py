"""CPU oracle for paged KV-cache decode attention (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The GPU library never does.
"""
