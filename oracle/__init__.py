"""CPU oracle for the k-quant weight matmul (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline legs of
``bench.py`` may import this package; the library never does.
"""
from .kq_oracle import *  # noqa: F401,F403
