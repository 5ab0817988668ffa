"""fp64 CPU oracle of the MoE decode-layer forward.

Test infrastructure only: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the product path.
"""
from .moe_oracle import *  # noqa: F401,F403
