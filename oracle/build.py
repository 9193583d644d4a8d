"""Build step for the FP64 CPU oracle (test infrastructure): gcc, no fused
multiply-add, no fast-math, OpenMP over rows.  Output: oracle/_build/liboracle.so."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "liboracle.so")
SOURCES = [os.path.join(HERE, "oracle.c"), os.path.join(HERE, "oracle.h")]


def commands(force=False):
    os.makedirs(BUILD, exist_ok=True)
    if not force and os.path.exists(LIB) and all(os.path.getmtime(s) <= os.path.getmtime(LIB) for s in SOURCES):
        return []
    return [(["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-shared",
              "-fPIC", "-o", LIB, SOURCES[0], "-lm"], LIB)]


def build(force=False):
    for argv, _ in commands(force):
        subprocess.run(argv, check=True)


if __name__ == "__main__":
    build(force=True)
