"""Compile the C oracle into ``oracle/liborc.so`` with the host gcc.

Test infrastructure only. The flags keep IEEE semantics: no fast-math and no
fused multiply-add contraction, because the oracle's FP32 accumulation is
specified as a rounded product followed by a rounded sum.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "fp8fg_oracle.c")
LIB = os.path.join(HERE, "liborc.so")


def build(force=False):
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
           "-fopenmp", "-shared", "-fPIC", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
