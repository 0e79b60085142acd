"""Build the sm_103a C-ABI library in-tree: csrc/*.cu -> _build/libhla.so.

Each translation unit compiles in parallel with nvcc for
``-gencode arch=compute_103a,code=sm_103a``; the objects link into one shared
library with the CUDA runtime linked statically, so the library loads without a
GPU (the CPU tests check its exports) and depends on nothing but libc/libstdc++.
"""

import os
import platform
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libhla.so")
SOURCES = ["api.cu", "kda.cu", "gemm.cu", "moe.cu", "layer.cu", "noalloc.cu", "tc_gemm.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _flags(extra=()):
    return ["-std=c++17", "-O3", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
            "-I", INCLUDE, "-I", CSRC, *extra]


def _deps():
    deps = [os.path.join(INCLUDE, "hla.h"), __file__]
    deps += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return deps


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def _stamp_ok():
    """Objects are reused only when they were built on this kind of machine."""
    try:
        with open(os.path.join(OUT, "BUILT_ON")) as f:
            return f.read().strip() == platform.machine()
    except OSError:
        return False


def build(force=False, verbose=False, extra_flags=()):
    """Compile (if stale) and return the path of libhla.so."""
    os.makedirs(OUT, exist_ok=True)
    if not _stamp_ok():
        force = True
    cc = nvcc()
    deps = _deps()
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        obj = os.path.join(OUT, src.replace(".cu", ".o"))
        if force or _stale(obj, [s] + deps):
            jobs.append([cc, *_flags(extra_flags), "-c", s, "-o", obj])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        return r.returncode

    if jobs:
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            codes = list(ex.map(run, jobs))
        if any(codes):
            raise RuntimeError("nvcc failed to compile the CUDA library")
    objs = [os.path.join(OUT, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or _stale(LIB, objs):
        cmd = [cc, "-shared", *ARCH, "-o", LIB + ".tmp", *objs]
        if run(cmd):
            raise RuntimeError("nvcc failed to link libhla.so")
        os.replace(LIB + ".tmp", LIB)
        with open(os.path.join(OUT, "BUILT_ON"), "w") as f:
            f.write(platform.machine())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
