"""CPU oracle of the MoE routing-and-expert step -- test infrastructure only.

Only the tests, `__graft_entry__.smoke()` and the benchmark's CPU-baseline leg
may import this package.  The library never routes work through it.
"""
from .moe_oracle import *  # noqa: F401,F403
