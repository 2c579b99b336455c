"""CPU oracle for the MoE / MoD layer hot path (test infrastructure only)."""
from .moe_oracle import *  # noqa: F401,F403
