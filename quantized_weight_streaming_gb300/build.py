"""Build step of libkq: every translation unit compiled in parallel by nvcc
for sm_103a only, then linked into quantized_weight_streaming_gb300/_build/libkq.so."""
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libkq.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["kq_host.cpp", "kq_prep.cu", "kq_stream.cu", "kq_tcs.cu", "kq_tc.cu", "kq_control.cu", "kq_direct.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("kq_internal.h", "kq_device.cuh", "kq_tc.h", "kq_stream.cuh", "kq_tcgen05.cuh")] + [os.path.join(INCLUDE, "kq.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _obj(src):
    return os.path.join(BUILD, os.path.splitext(src)[0] + ".o")


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force=False, verbose_ptxas=False):
    os.makedirs(BUILD, exist_ok=True)
    procs = []
    for src in SOURCES:
        path = os.path.join(CSRC, src)
        obj = _obj(src)
        if force or _stale(obj, [path] + HEADERS):
            argv = ["nvcc", *ARCH, *COMMON, "-c", path, "-o", obj]
            if verbose_ptxas and src.endswith(".cu"):
                argv += ["-Xptxas", "-v"]
            procs.append((subprocess.Popen(argv), argv))
    failed = [argv for p, argv in procs if p.wait() != 0]
    if failed:
        raise RuntimeError("nvcc failed: " + " ".join(failed[0]))
    objs = [_obj(s) for s in SOURCES]
    if force or procs or _stale(LIB, objs):
        subprocess.run(["nvcc", *ARCH, "-shared", "-cudart", "shared", "-o", LIB, *objs], check=True)
    return LIB


if __name__ == "__main__":
    build(force=True, verbose_ptxas="-v" in sys.argv)
