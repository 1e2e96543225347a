"""CPU oracles for the routed MoE layer: test infrastructure, not the product.

moe_oracle.cpp (loaded through cpp_oracle.py) is the C++ float64 statement of the
layer; moe_oracle.py is the same definition in float64 numpy, and the pins run
against both.  Only the tests, the package's smoke check and the benchmark's CPU
legs use them.  The CUDA library never imports, links or calls anything here.
"""
from .moe_oracle import *  # noqa: F401,F403
from . import moe_oracle  # noqa: F401
