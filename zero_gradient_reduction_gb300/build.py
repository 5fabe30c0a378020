"""Builds libzr.so (the C-ABI library) in-tree with nvcc for sm_103a.

Translation units compile in parallel; the host file and the host side of the .cu files
are built with -ffp-contract=off and the device side with -fmad=false, so no fp32
multiply-add is fused anywhere on the path (the kernels also use explicit _rn intrinsics).
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libzr.so")
ARCH = os.environ.get("ZR_CUDA_ARCH", "103a")

CU = ["zr_step.cu", "zr_inplace.cu", "zr_collectives.cu", "zr_noalloc.cu", "zr_zero3.cu", "zr_offload.cu"]
CPP = ["zr_host.cpp", "zr_offload_host.cpp"]
# the host AdamW of ZeRO-Offload: vectorised (no errno on sqrt), still one rounding per op
CPP_EXTRA = {"zr_offload_host.cpp": ["-O3", "-fno-math-errno", "-pthread"]}
# every header a translation unit may include: a change to any of them rebuilds all units
HEADERS = [os.path.join(INCLUDE, "zr.h")] + sorted(
    os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh")))


def _nvcc_flags(verbose_ptxas: bool = False):
    f = [f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}", "-O3", "-lineinfo", "-std=c++17", "-fmad=false",
         "-Xcompiler", "-fPIC,-ffp-contract=off,-O2", f"-I{INCLUDE}", f"-I{CSRC}"]
    if verbose_ptxas:
        f += ["-Xptxas", "-v"]
    return f


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, verbose_ptxas: bool):
    path = os.path.join(CSRC, src)
    obj = os.path.join(OBJ, src + ".o")
    if not _stale(obj, [path] + HEADERS) and not verbose_ptxas:
        return obj, ""
    if src.endswith(".cu"):
        cmd = ["nvcc", "-c", path, "-o", obj] + _nvcc_flags(verbose_ptxas)
    else:
        cmd = ["g++", "-c", path, "-o", obj, "-O2", "-std=c++17", "-fPIC", "-ffp-contract=off", f"-I{INCLUDE}",
               f"-I{CSRC}"] + CPP_EXTRA.get(src, [])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"compile failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return obj, r.stdout + r.stderr


def build(force: bool = False, verbose_ptxas: bool = False) -> str:
    os.makedirs(OBJ, exist_ok=True)
    srcs = CU + CPP
    if force:
        for s in srcs:
            o = os.path.join(OBJ, s + ".o")
            if os.path.exists(o):
                os.remove(o)
    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose_ptxas), srcs))
    objs = [r[0] for r in results]
    if verbose_ptxas:
        for s, (_, log) in zip(srcs, results):
            if log:
                sys.stdout.write(f"--- {s}\n{log}")
    if force or _stale(LIB, objs):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = ["nvcc", "-shared", "-cudart", "shared", f"-gencode=arch=compute_{ARCH},code=sm_{ARCH}", "-o", tmp] + \
            objs + ["-lpthread"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv)
    print(LIB)
