"""Compile the CPU oracle into oracle/_fp8rl_oracle.so (test infrastructure).

Plain g++, no CUDA, no fast-math, no FMA contraction, so that each binary32 /
float64 operation in the oracle is one IEEE operation rounded to nearest-even
on both x86-64 and aarch64 hosts.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp8rl_oracle.cpp")
LIB = os.path.join(HERE, "_fp8rl_oracle.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-pthread", SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
