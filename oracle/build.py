"""Compile the CPU oracle (rcc_oracle.cpp) into oracle/liboracle_rcc.so.

Test infrastructure: the oracle is built so the tests, the smoke check and the
benchmark's CPU-baseline leg can load it.  Plain g++, -O2, no fast-math and no
floating-point contraction, so each fp32 operation is rounded once in the order
the source writes it, on x86-64 and aarch64 alike.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "rcc_oracle.cpp")
LIB = os.path.join(HERE, "liboracle_rcc.so")

CXXFLAGS = ["-std=c++17", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
            "-fno-fast-math", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC),
                                              os.path.getmtime(os.path.join(HERE, "rcc_oracle.h")))):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["g++", *CXXFLAGS, SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
