"""Oracle for the boundary-quantised GCN aggregation.

TEST INFRASTRUCTURE ONLY.  Plain, slow CPU code (numpy/scipy, fp64
accumulation) that states what the GPU library computes.  Only the test suite,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import it; the library never does, and shares no code with it.
"""
from .oracle import *  # noqa: F401,F403
