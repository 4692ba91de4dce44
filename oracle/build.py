"""Compile the fp64 CPU oracle into a shared library (test infrastructure only).

The oracle is plain C99 + pthreads + libm, built with gcc at -O2 and without
-ffast-math so that every exp, tanh, product and sum keeps IEEE fp64 semantics.
"""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "ua_oracle.c")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libua_oracle.so")


def build(force: bool = False) -> str:
    """Build ``libua_oracle.so`` if it is missing or older than its source."""
    os.makedirs(OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= os.path.getmtime(SRC)):
        return LIB
    tmp = LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared", "-pthread",
           "-D_POSIX_C_SOURCE=200809L", "-o", tmp, SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True))
