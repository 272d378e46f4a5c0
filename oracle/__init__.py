"""CPU oracle for the NF4 + double-quantized LoRA linear layer (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` import this package. The GPU library never does.
"""
