"""Build the CPU oracle (oracle.c -> liboracle.so) with the host C compiler.

TEST INFRASTRUCTURE ONLY: the oracle is the checker for the CUDA path, so it is
built beside it, but nothing on the product path loads it.

Built without FP contraction (-ffp-contract=off) so every fp64 product and sum
in the materialisation is rounded once, in the stated order. Portable C99, no
target-specific flags, so it builds the same on x86_64 and aarch64.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc, "-std=c99", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
