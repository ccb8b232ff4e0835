"""fp64 CPU oracle of the MoE layer forward.  Test infrastructure only: used by
tests/, __graft_entry__.smoke() and bench.py's CPU-baseline leg, never by the
product path."""
from .moe_oracle import *  # noqa: F401,F403
