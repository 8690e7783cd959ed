"""Compile the CPU oracle (test infrastructure) into ``oracle/liboracle.so``.

The flags keep the compiler from fusing or reordering anything: no FMA contraction, no
fast-math, IEEE division. The only fused operations are the ones the source spells out
(the exact quantiser product in double, and fmaf for each term of the hop sums).
OpenMP only parallelises independent blocks and receivers.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "zpp_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

BASE_FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-frounding-math",
              "-fPIC", "-shared", "-Wall"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)
            and os.path.getmtime(LIB) >= os.path.getmtime(__file__)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", *BASE_FLAGS, "-fopenmp", SRC, "-o", tmp, "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:  # no OpenMP runtime: build single-threaded
        cmd = ["gcc", *BASE_FLAGS, SRC, "-o", tmp, "-lm"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("oracle build failed:\n" + r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
