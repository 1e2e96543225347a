"""CPU oracle for the routed MoE layer: test infrastructure, not the product.

Only the tests, the package's smoke check and the benchmark's CPU-baseline leg
use it.  The CUDA library never imports, links or calls anything here.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
