"""Compile the CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain gcc, no fused multiply-add contraction, no fast-math: the oracle's fp32
operation sequence defines the compressed-cache bytes exactly.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "dsv4_oracle.c")
HDR = os.path.join(HERE, "dsv4_oracle.h")
LIB = os.path.join(HERE, "liboracle.so")


def build_oracle(force: bool = False) -> str:
    """Build liboracle.so if missing or older than its sources; return its path."""
    if not force and os.path.exists(LIB):
        lib_m = os.path.getmtime(LIB)
        if lib_m >= os.path.getmtime(SRC) and lib_m >= os.path.getmtime(HDR):
            return LIB
    tmp = LIB + ".%d.tmp" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-Wall", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
