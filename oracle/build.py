"""Compile the float64 CPU oracle (test infrastructure) into oracle/liboracle.so.

Plain gcc, no CUDA: the oracle shares nothing with the GPU library. The build
is quick (one C file) and is redone whenever the source is newer than the
shared object, so tests and the benchmark can call `ensure_built()` freely.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "gdr_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(src=SRC, out=LIB, extra_flags=()):
    """Compile `src` into the shared object `out` and return its path."""
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-pthread", "-std=c11", *extra_flags,
           "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def ensure_built():
    """Build liboracle.so when it is missing or older than its source."""
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        build()
    return LIB


if __name__ == "__main__":
    print(build())
    sys.exit(0)
