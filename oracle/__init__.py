"""fp64 CPU oracle of the MoE layer and its MXFP8 codec.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. The product path never
does.

Parity pins: every function here is checked by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against values fixed by the pages or by mathematics
(closed forms, finite differences, brute force, library routines, spec values).
The only function without such a pin is the optional SwiGLU clamp, which the
oracle does not implement (parity unpinned; the library rejects it).
"""
