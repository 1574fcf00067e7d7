"""CPU oracle for the BASTION draft-tree hot path -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding) never calls it.
"""
from .oracle import *  # noqa: F401,F403
