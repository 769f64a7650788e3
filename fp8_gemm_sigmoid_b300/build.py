"""Build libmoe.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Usage: python -m fp8_gemm_sigmoid_b300.build [--force] [--verbose] [--checks]

--checks builds libmoe_checks.so instead: the same sources with -DMOE_CHECKS, whose kernels
check the indices callers pass in and record failures in the device error word (a debug
build; the hot path is libmoe.so).
"""
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libmoe.so")
CHECKS_LIB = os.path.join(HERE, "libmoe_checks.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-cudart", "shared",
]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.h")) +
                              glob.glob(os.path.join(CSRC, "*.cuh")) +
                              [os.path.join(ROOT, "include", "moe.h")])


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force=False, verbose=False, checks=False):
    """Compile every .cu under csrc/ into libmoe.so, or with checks=True into
    libmoe_checks.so with -DMOE_CHECKS (one nvcc call per object, then link)."""
    lib = CHECKS_LIB if checks else LIB
    if not force and up_to_date(lib):
        return lib
    objdir = os.path.join(HERE, "_build_checks" if checks else "_build")
    os.makedirs(objdir, exist_ok=True)
    objs = []
    procs = []
    for src in sources():
        obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
        cmd = [NVCC, *NVCC_FLAGS, *(["-DMOE_CHECKS"] if checks else []), "-I", os.path.join(ROOT, "include"),
               "-c", src, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = False
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or p.returncode != 0):
            sys.stdout.write(out.decode())
        if p.returncode != 0:
            failed = True
            sys.stdout.write("nvcc failed on %s\n" % src)
    if failed:
        raise RuntimeError("libmoe build failed")
    tmp = lib + ".tmp%d" % os.getpid()
    link = [NVCC, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-cudart", "shared",
            "-Xlinker", "--no-undefined",
            *objs, "-o", tmp]
    subprocess.run(link, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv, checks="--checks" in sys.argv))
