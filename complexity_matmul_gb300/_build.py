"""Build ``liblcgemm`` in-tree with nvcc for sm_103a (no cmake, no torch extension).

Each ``csrc/*.cu`` translation unit is compiled in parallel, then linked into
``complexity_matmul_gb300/_build/liblcgemm.<machine>.so`` (the machine suffix
keeps x86_64 and aarch64 builds apart).  A unit is recompiled when it or any
header it may include is newer than its object.
"""
from __future__ import annotations

import glob
import os
import platform
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
MACHINE = platform.machine()
LIB = os.path.join(BUILD, f"liblcgemm.{MACHINE}.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC",
         "-Xcompiler", "-Wall", "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build liblcgemm")


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    hdr_time = max([os.path.getmtime(p) for p in _headers()] + [0.0])

    def obj_of(src):
        return os.path.join(BUILD, os.path.basename(src)[:-3] + f".{MACHINE}.o")

    def compile_one(src):
        obj = obj_of(src)
        if not force and os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(src), hdr_time):
            return obj, None
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            return obj, f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}"
        os.replace(obj + ".tmp", obj)
        return obj, (r.stdout + r.stderr) if verbose else None

    srcs = sources()
    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    errors = [msg for _, msg in results if msg and "error" in msg.lower()]
    if errors:
        raise RuntimeError("liblcgemm compilation failed:\n" + "\n".join(errors))
    if verbose:
        for _, msg in results:
            if msg:
                print(msg)
    objs = [o for o, _ in results]
    if force or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        cmd = [nvcc, *ARCH, "-shared", "-o", LIB + ".tmp", *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"liblcgemm link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
