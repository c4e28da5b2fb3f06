"""CPU oracle for the skinny quantized linear -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s cpu_baseline and
``--impl reference`` legs may import this package.
"""
