"""Plain fp64 CPU oracle of the fused MoE forward -- test infrastructure.

Only tests/, ``__graft_entry__.smoke()`` and bench.py's CPU-baseline legs
import this package; the CUDA product path never does.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import __all__  # noqa: F401
