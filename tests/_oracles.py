"""The two CPU oracles the pins run against: the float64 numpy statement
(oracle/moe_oracle.py) and the C++ float64 one (oracle/moe_oracle.cpp)."""
from oracle import cpp_oracle
from oracle import moe_oracle

NAMES = ["numpy", "cpp"]


def get(name):
    return moe_oracle if name == "numpy" else cpp_oracle.default()
