"""CPU oracle for token-level KV selection (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
and reference legs may import this package. The product path never calls it.
"""
from .tokenselect_oracle import *  # noqa: F401,F403
