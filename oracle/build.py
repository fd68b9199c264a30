"""Compile the C oracle (``pa_oracle.c``) into ``liboracle.so`` with gcc.

Test infrastructure: see the header of ``oracle/__init__.py``.
"""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "pa_oracle.c")
LIB = os.path.join(HERE, "liboracle.so")


def build(src=SRC, out=LIB, extra=()):
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", *extra, src, "-o", out, "-lm"]
    subprocess.run(cmd, check=True)
    return out


def ensure_built():
    if not os.path.exists(LIB) or os.path.getmtime(LIB) < os.path.getmtime(SRC):
        build()
    return LIB


if __name__ == "__main__":
    print(build(*sys.argv[1:2]))
