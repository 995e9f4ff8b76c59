"""Float64 CPU oracle (test infrastructure only; never on the product path).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.
"""
