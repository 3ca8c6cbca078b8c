"""Build the oracle's shared library (liboracle.so) with the host C compiler.

Test infrastructure only.  The flags keep IEEE semantics: no -ffast-math and
no floating-point contraction, so the sequential fp64 loops in oracle.c run
exactly in the order they are written.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")

CFLAGS = ["-O2", "-fPIC", "-shared", "-std=c11", "-fno-fast-math",
          "-ffp-contract=off", "-Wall", "-Wextra"]


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/liboracle.so if it is missing or stale."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(SRC),
                                             os.path.getmtime(os.path.join(HERE, "oracle.h")))):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.run([cc, *CFLAGS, "-o", tmp, SRC, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv))
