"""FP64 CPU oracle for triangular attention: test infrastructure only.

Imported by ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg, never by the product package.
"""
