"""fp64 CPU oracle of the vocabulary cross-entropy (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
use this package.  See ``ce_oracle`` for the definitions and their sources.
"""
from .ce_oracle import *  # noqa: F401,F403
from . import ce_oracle, rounding  # noqa: F401
