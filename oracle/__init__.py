"""CPU oracle of the MoE layer (float64, numpy).

TEST INFRASTRUCTURE ONLY: imported by tests/, __graft_entry__.smoke() and the
bench's CPU-baseline / reference leg, never by the CUDA library or its binding."""
from .moe_oracle import *  # noqa: F401,F403
