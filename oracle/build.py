"""Compile the float64 oracle (oracle.c, linattn.c) into oracle/liboracle.so.

Test infrastructure: the oracle is built so the tests and the benchmark's
CPU-baseline leg can call it; the CUDA library never links or loads it.
Flags: -O2, no -ffast-math (IEEE double arithmetic and libm exp must be kept),
no -march=native (the .so may run on a different host than the one that
built it).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRCS = [os.path.join(HERE, "oracle.c"), os.path.join(HERE, "linattn.c")]
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False) -> str:
    """Build liboracle.so if it is missing or older than its sources; return its path."""
    if (not force and os.path.exists(LIB)
            and all(os.path.getmtime(LIB) >= os.path.getmtime(s) for s in SRCS)):
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fno-fast-math",
           "-o", tmp, *SRCS, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
