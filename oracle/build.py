"""Build the C++ oracle (oracle/moe_oracle.cpp) into oracle/libmoe_oracle.so.

    python -m oracle.build

Test infrastructure: the CUDA library never links or loads it.  Plain g++ with
generic x86-64 code (no -march), -O2, and no contraction of a*b+c into fused
multiply-adds, so each product and sum rounds as the source states.  `plant`
builds a variant with one deliberate mistake (the tests' planted slips) into a
directory of the caller's choosing.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
LIB = os.path.join(HERE, "libmoe_oracle.so")
FLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-ffp-contract=off", "-pthread"]


def build(out: str = LIB, plant: int = 0, force: bool = False) -> str:
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(SRC):
        return out
    cmd = [os.environ.get("CXX", "g++"), *FLAGS, f"-DORC_PLANT={int(plant)}", SRC, "-o", out + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("g++ failed on the C++ oracle")
    os.replace(out + ".tmp", out)
    return out


if __name__ == "__main__":
    print(build(force="-f" in sys.argv))
