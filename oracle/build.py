"""Compile the fp64 CPU oracle (conv_ref.c) into liboracle.so.

TEST INFRASTRUCTURE: the oracle is only used by the tests, the smoke check and
the bench's CPU-baseline leg. Plain gcc; OpenMP when the compiler has it.
FMA contraction is off so the oracle rounds the same way on x86 and Arm.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "conv_ref.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Build liboracle.so next to this file if it is missing or stale."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    base = ["gcc", "-std=c99", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
            SRC, "-o", LIB + ".tmp"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
