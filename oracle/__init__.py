"""fp64 CPU oracle of the KATA causal normalised linear-attention forward.

Test infrastructure only: used by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the product path.
"""
from .kata_oracle import *  # noqa: F401,F403
from .kata_oracle import SCAN_SEQUENTIAL, SCAN_TREE  # noqa: F401
