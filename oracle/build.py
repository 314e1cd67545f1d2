"""Build the CPU oracle (``oracle/liboracle.so``) with gcc.

Test infrastructure: only the test-suite, the smoke check and the benchmark's
CPU-baseline leg load the result.  ``-ffp-contract=off`` keeps gcc from
fusing a*b+c on targets where FMA is part of the base ISA (aarch64), so the
only fused multiply-add is the explicit ``fmaf`` of the combine.
"""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
HDR = os.path.join(HERE, "oracle.h")
LIB = os.path.join(HERE, "liboracle.so")

BASE_FLAGS = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared", "-Wall"]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in (SRC, HDR, __file__))


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile liboracle.so if missing or older than its sources; return its path."""
    if not force and not _stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *BASE_FLAGS, "-fopenmp", SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        # no libgomp on this host: the pragmas are ignored and the oracle runs on one thread
        cmd = ["gcc", *BASE_FLAGS, SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("oracle build failed: " + " ".join(cmd))
    if verbose:
        print(" ".join(cmd))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
