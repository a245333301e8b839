"""CPU oracle for masked attention in the column-wise sparse mask form.

TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path imports,
calls or links this package: only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use it.  It shares
no code, table or helper with the CUDA library, and the library never falls
back to it.

What it computes, from the pages and the plain definitions:

* ``oracle.masks`` - the mask predicate written out densely, the exact count of
  visible score entries, the empty/full/partial tile rule evaluated column by
  column, the per-tile work lists, the longest-first unit order and the
  clip/shift/max localisation of the bounds to a rank's query chunks;
* ``oracle.attention`` - exact scaled-dot-product attention under the mask and
  its gradients, in float64, on the bf16-rounded inputs.

Every function names the passage it follows.  Parity pins live in
``tests/test_oracle_*.py``.
"""
from . import masks, attention  # noqa: F401
