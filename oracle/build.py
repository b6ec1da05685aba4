"""Compile the CPU oracle (TEST INFRASTRUCTURE) into oracle/libagoq_oracle.so
and, where the compiler supports OpenMP, an all-core build of the same source
into oracle/libagoq_oracle_omp.so.

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
LIB_OMP = os.path.join(HERE, "libagoq_oracle_omp.so")

CFLAGS = ["-O2", "-ffp-contract=off", "-fno-fast-math", "-std=c11", "-fPIC", "-shared",
          "-Wall", "-Wextra"]


def _compile(target, extra, force):
    if (not force and os.path.exists(target)
            and os.path.getmtime(target) >= max(os.path.getmtime(SRC), os.path.getmtime(__file__))):
        return target
    tmp = target + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, *extra, "-o", tmp, SRC, "-lm"], check=True)
    os.replace(tmp, target)
    return target


def build(force: bool = False) -> str:
    """Build the single-threaded oracle library (and, if possible, the all-core
    one) if missing or older than the source; return the single-threaded path."""
    _compile(LIB, ["-Wno-unknown-pragmas"], force)
    build_omp(force)
    return LIB


def build_omp(force: bool = False):
    """The all-core build (OpenMP), or None if the compiler cannot build it."""
    try:
        return _compile(LIB_OMP, ["-fopenmp"], force)
    except (subprocess.CalledProcessError, OSError):
        return None


if __name__ == "__main__":
    print(build(force="--force" in sys.argv), build_omp())
