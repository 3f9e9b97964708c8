"""CPU oracle of the fused quantised linear layer (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package; the CUDA path never does.
"""
