"""CPU oracle of the dropless MoE layer (test infrastructure only).

Plain, slow, fp64 NumPy.  It shares no code with the CUDA library and neither
imports the other.  Only the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may use it; the product path never does.
"""
from .moe_oracle import *  # noqa: F401,F403
