"""Compile the CPU oracle (TEST INFRASTRUCTURE) into oracle/libagoq_oracle.so.

The flags matter: -ffp-contract=off keeps every multiply and add a separately
rounded binary32 operation (aarch64 GCC fuses them by default), and no
fast-math option is given, so subnormals, signed zeros and IEEE division are
kept.  Run directly (``python oracle/build.py``) or through the package build.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "agoq_oracle.c")
LIB = os.path.join(HERE, "libagoq_oracle.so")

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Build the oracle library if it is missing or older than its source."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = ["gcc", *CFLAGS, "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
