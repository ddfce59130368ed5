"""CPU oracle of the CSA2 global-attention step (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` import this package; the CUDA library never does.
"""
from . import csa2_oracle  # noqa: F401
