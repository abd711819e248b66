"""CPU oracle of the MoE layer -- test infrastructure only.

Imported only by the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline / reference legs. The library never imports or calls it, and it
shares no code with the CUDA path.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
