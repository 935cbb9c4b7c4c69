"""Compile the fp64 CPU oracle (``dust_oracle.c``) into ``libdust_oracle.so``.

Test infrastructure: the oracle is the checker, never part of the product
path. Portable C11 (no architecture flags), so the same source builds on the
x86_64 development host and on the aarch64 GPU host.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dust_oracle.c")
LIB = os.path.join(HERE, "libdust_oracle.so")


def build(force: bool = False) -> str:
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-fPIC", "-shared",
           "-fvisibility=hidden", "-Wall", "-Wextra", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
