"""CPU oracles for the k-quant and TQ4_1S weight matmuls (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package; the library never does.
"""
from .kq_oracle import *  # noqa: F401,F403
from . import tq4_oracle  # noqa: F401
