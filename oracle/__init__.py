"""CPU float64 oracle for the S4 layer forward path (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA path never calls it.
"""
from .s4_oracle import *  # noqa: F401,F403
