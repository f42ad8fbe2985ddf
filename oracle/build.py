"""Compile the fp64 CPU oracle (dsc_oracle.c) into oracle/libdsc_oracle.so.

Test infrastructure only: the product library never links or loads it.
Run as a script or call build_oracle().
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dsc_oracle.c")
LIB = os.path.join(HERE, "libdsc_oracle.so")


def build_oracle(force: bool = False) -> str:
    """Build the oracle shared library if it is missing or stale; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           "-Wextra", "-o", LIB + ".tmp", SRC]
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force="--force" in sys.argv))
