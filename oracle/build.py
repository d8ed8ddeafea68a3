"""Compiles the oracle's C scan into oracle/libkda_oracle.so with gcc.

TEST INFRASTRUCTURE: the library built here is loaded only by tests/,
__graft_entry__.smoke() and bench.py's CPU-baseline leg.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "kda_scan.c")
LIB = os.path.join(HERE, "libkda_oracle.so")


def build(force: bool = False) -> str:
    """Builds the shared library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-D_GNU_SOURCE",
           SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
