"""Compile the float64 CPU oracle (oracle.c) into liboracle.so beside it.

Test infrastructure only: the oracle is the checker the CUDA library is compared
against.  Plain gcc, -O2, OpenMP when the compiler supports it.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(force: bool = False, quiet: bool = True) -> str:
    """Build liboracle.so if missing or older than oracle.c; return its path."""
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    cc = os.environ.get("CC", "gcc")
    tmp = LIB + ".tmp%d" % os.getpid()
    cmd = [cc, "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", SRC, "-o", tmp, "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError("oracle build failed:\n%s\n%s" % (" ".join(cmd), res.stderr))
    os.replace(tmp, LIB)
    if not quiet:
        print(" ".join(cmd))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, quiet=False))
