"""CPU oracle for the routed MoE FFN forward (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may import this package.  The product path (the C-ABI
library and its Python binding) never calls it and shares no code with it.
"""
from .moe_oracle import *  # noqa: F401,F403
