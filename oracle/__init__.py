"""CPU fp64 oracle for exact attention: TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package.  The
CUDA library and its Python binding never import it, and it imports nothing
from them.

Modules:
  attention  -- the plain definition in float64 (forward, backward, merge of
                results over disjoint key sets).
  blockwise  -- an fp64 restatement of the tiled FlashAttention-2 forward
                algorithm, used only to check the algorithm against the
                definition on the CPU.

Pins: every function here is checked in ``tests/test_oracle.py`` against
closed forms, invariants, brute force on tiny inputs, finite differences and
the counts printed on the pages; ``tests/test_oracle_mutants.py`` plants
mistakes in it and checks that a pin catches each.  No function is
unpinned.
"""
from . import attention, blockwise  # noqa: F401
