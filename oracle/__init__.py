"""fp64 CPU oracle of the MoE layer and its MXFP8 codec.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package. The product path never
does.

Parity pins: every function here is checked by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against values fixed by the pages or by mathematics
(closed forms, finite differences, brute force, library routines, spec values),
the swiglu_limit clamp and the shared output gate included (central finite
differences of every gradient with the clamp active, a single unit worked by
hand, and a limit too large to bind leaving the layer unchanged).
"""
