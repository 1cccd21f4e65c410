"""Test infrastructure: the fp64 CPU oracle for quantized-KV decode attention.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline and
reference legs may import this package.  The product path never does.
"""
