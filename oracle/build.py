"""Build the CPU oracle shared library (plain g++, portable: x86_64 and aarch64).

Test infrastructure: only the tests, the smoke check and the benchmark's CPU-baseline
leg load the result.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_oracle.cpp")
LIB = os.path.join(HERE, "libmoe_oracle.so")

FLAGS = ["-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
         "-ffp-contract=off", "-fno-fast-math", "-fno-finite-math-only"]


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cmd = ["g++", *FLAGS, SRC, "-o", LIB + ".tmp"]
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
