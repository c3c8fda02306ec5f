"""Compile the CPU oracle (ufp4_oracle.c) into oracle/libufp4_oracle.so.

Test infrastructure only: the oracle is the checker for the CUDA library,
never part of it.  Plain gcc, no vectorisation flags that change rounding:
-ffp-contract=off keeps every fp32 step a single IEEE rounding on both x86-64
and aarch64 (gcc contracts a*b+c into FMA by default on aarch64).
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ufp4_oracle.c")
LIB = os.path.join(HERE, "libufp4_oracle.so")
FLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-fPIC", "-shared"]


def build_oracle(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    subprocess.check_call(["gcc", *FLAGS, "-o", tmp, SRC, "-lm"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
