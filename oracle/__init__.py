"""Oracle for the fused APL MoE layer: TEST INFRASTRUCTURE ONLY.

A plain, slow, obviously correct CPU restatement (numpy, fp64) of what the
hot path computes, written from the PagedWeight pages' description of the
method ("Paged Weight Representation" and "Fused Mixed-Precision Kernel" in
the core components of the technical summaries; the paper abstract) and the
layout fixed for this build (n packed bit-planes, MSB first, along K per
output row; per-row, per-bitwidth fp16 lookup tables).

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  It shares
no code with the CUDA path and imports nothing from it; the product must
never call it.

Modules:
  apl    -- bit-plane pack/unpack, child LUTs, dequantisation
  moe    -- routing, permutation, expert MLP, combine, whole layer

Parity status: every function here is pinned by tests/test_oracle_*.py
(hand-derived golden fixtures, closed forms, invariants, brute force and
independent library routines), except the child-LUT construction rule, which
is this build's own reading of "associated lookup tables" and is pinned only
by its own definition (parity unpinned with respect to the pages).
"""
from . import apl, moe  # noqa: F401
