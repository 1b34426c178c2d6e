"""Compile libspecverify.so (the CUDA kernels and the C ABI) for sm_103a."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SOURCES = [os.path.join(HERE, "csrc", "spec_verify.cu"), os.path.join(HERE, "csrc", "kv_commit.cu"),
           os.path.join(HERE, "csrc", "lmhead.cu")]
DEPENDS = SOURCES + [os.path.join(HERE, "csrc", "sv_device.cuh"), os.path.join(HERE, "csrc", "sv_tc.cuh"),
                     os.path.join(ROOT, "include", "spec_verify.h")]
LIBRARY = os.path.join(HERE, "libspecverify.so")
NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
              "-Xcompiler", "-fPIC"]


def nvcc() -> str:
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    cand = os.path.join(home, "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def stale() -> bool:
    if not os.path.exists(LIBRARY):
        return True
    t = os.path.getmtime(LIBRARY)
    return any(os.path.getmtime(f) > t for f in DEPENDS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles the translation units in parallel, then links the library."""
    if not force and not stale():
        return LIBRARY
    tag = f".tmp{os.getpid()}"
    objs, procs = [], []
    for src in SOURCES:
        obj = os.path.splitext(src)[0] + tag + ".o"
        cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-c", "-o", obj, src]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
            print(" ".join(cmd), file=sys.stderr)
        objs.append(obj)
        procs.append(subprocess.Popen(cmd))
    try:
        bad = [p.args for p in procs if p.wait() != 0]
        if bad:
            raise subprocess.CalledProcessError(1, bad[0])
        tmp = LIBRARY + tag
        subprocess.run([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-o", tmp, *objs],
                       check=True)
        os.replace(tmp, LIBRARY)
    finally:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIBRARY


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
