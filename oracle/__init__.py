"""CPU oracle of the MoE expert layer -- TEST INFRASTRUCTURE, not product code.

A plain, slow, float64 restatement of what the layer computes, written from
the pages' description and the layer's fixed formulas.  Only ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import it.  It shares no code with the CUDA library (no kernels, headers,
tables or helpers) and neither imports the other.

Every function is pinned in ``tests/test_oracle_*.py`` to something other than
itself: hand-computed encodings (``tests/golden/``), brute force on small
inputs, closed forms and invariants.
"""
from . import bfp8, formats, moe  # noqa: F401
