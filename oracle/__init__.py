"""CPU oracle of the tensor-parallel MLP sublayer -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never does.
"""
from . import tpmlp_oracle  # noqa: F401
