"""CPU oracle of the W4A16 MoE grouped GEMM -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg / reference arm may import, call or execute anything in this package. The
CUDA library never imports it and shares no code with it.
"""

from .moe_oracle import *  # noqa: F401,F403
