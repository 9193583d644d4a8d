"""Build step for the synthetic input generator: a host library (gcc) and its
device twin (nvcc, sm_103a).  Both land in synth/_build/."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
HOST_LIB = os.path.join(BUILD, "libsynth_host.so")
DEV_LIB = os.path.join(BUILD, "libsynth_dev.so")


def _newer(target, sources):
    if not os.path.exists(target):
        return False
    t = os.path.getmtime(target)
    return all(os.path.getmtime(s) <= t for s in sources)


def commands(force=False):
    """Return the compile commands still needed, as (argv, output) pairs."""
    os.makedirs(BUILD, exist_ok=True)
    hdr = os.path.join(HERE, "philox.h")
    out = []
    src = os.path.join(HERE, "gen_host.c")
    if force or not _newer(HOST_LIB, [src, hdr]):
        out.append((["gcc", "-O2", "-std=c11", "-fopenmp", "-shared", "-fPIC", "-o", HOST_LIB, src], HOST_LIB))
    src = os.path.join(HERE, "gen_device.cu")
    if force or not _newer(DEV_LIB, [src, hdr]):
        out.append((["nvcc", "-O3", "-std=c++17", "-gencode", "arch=compute_103a,code=sm_103a", "-lineinfo",
                     "-shared", "-Xcompiler", "-fPIC", "-o", DEV_LIB, src], DEV_LIB))
    return out


def build(force=False):
    procs = [(subprocess.Popen(argv), argv) for argv, _ in commands(force)]
    for p, argv in procs:
        if p.wait() != 0:
            raise RuntimeError("build failed: " + " ".join(argv))


if __name__ == "__main__":
    build(force=True)
