"""Builds ``liboracle.so`` from ``oracle.c`` (test infrastructure only).

The oracle is plain C compiled by the host compiler.  OpenMP is used when the
compiler supports it; it only spreads independent output units over cores.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build_oracle(force: bool = False) -> str:
    """Compile the oracle if the shared object is missing or older than its source."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build_oracle(force=True))
