"""CPU oracle for the compressed-KV decode step (test infrastructure).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package.  It shares no code with the CUDA
library or its binding and imports nothing from them.
"""
from .kvc_oracle import *  # noqa: F401,F403
