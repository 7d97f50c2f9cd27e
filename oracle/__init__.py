"""CPU oracle of the sparse MoE layer (test infrastructure; see moe_oracle.py)."""
from .moe_oracle import *  # noqa: F401,F403
