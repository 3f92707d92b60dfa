"""Compile the float64 CPU oracle (oracle.c) into liborc.so with gcc.

TEST INFRASTRUCTURE: the oracle is used only by the tests, the smoke check and
the CPU-baseline leg of the benchmark. The CUDA library never links it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liborc.so")


def build(force: bool = False) -> str:
    """Build liborc.so next to oracle.c if it is missing or older than the source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    # -ffp-contract=off: no fused multiply-add contraction, so x86 and Arm hosts
    # round every product and sum the same way.
    cmd = ["gcc", "-O2", "-std=c99", "-D_POSIX_C_SOURCE=200809L", "-ffp-contract=off",
           "-fPIC", "-shared", SRC, "-o", tmp, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
