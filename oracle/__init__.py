"""The fp64 CPU oracle of the MLA attention forward (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
may import this package.  The CUDA library never does.
"""
from .mla_oracle import *  # noqa: F401,F403
