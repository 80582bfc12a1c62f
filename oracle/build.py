"""Compile the C oracle into ``oracle/liboracle.so`` with the host gcc.

Test infrastructure: the product path never runs this.  The flags keep the
oracle's arithmetic literal: no fused multiply-add contraction, no fast-math
reassociation, no flush-to-zero.
"""

from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")
FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
         "-Wall", "-Wextra"]
# Row loops shared among threads (results do not depend on the count); the
# build falls back to one thread where the compiler has no OpenMP runtime.
OPENMP = ["-fopenmp"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIBRARY)
            and os.path.getmtime(LIBRARY) >= max(os.path.getmtime(SOURCE), os.path.getmtime(__file__))):
        return LIBRARY
    tmp = LIBRARY + f".tmp{os.getpid()}"
    cc = os.environ.get("CC", "gcc")
    res = subprocess.run([cc, *FLAGS, *OPENMP, SOURCE, "-o", tmp, "-lm"], capture_output=True, text=True)
    if res.returncode != 0:
        subprocess.run([cc, *FLAGS, SOURCE, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
