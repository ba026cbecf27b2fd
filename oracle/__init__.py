"""CPU oracle of the latent-MoE layer forward (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline and
reference legs may import this package; the CUDA library never does.
"""
from .lmoe_oracle import *  # noqa: F401,F403
from . import lmoe_oracle  # noqa: F401
