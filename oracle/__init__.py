"""fp64 CPU oracle for exact tiled attention forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference leg may import this package. It shares no code with the CUDA path.
"""
from .oracle import *  # noqa: F401,F403
from .oracle import build, attention, attention_head, attention_rows, blockwise_attention  # noqa: F401
