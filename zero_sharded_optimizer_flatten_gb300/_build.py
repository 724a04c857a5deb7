"""Build libzero.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into
zero_sharded_optimizer_flatten_gb300/libzero.so.  No cmake, no torch
extension machinery: the library has a plain C ABI and no torch types.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libzero.so")

SOURCES = ["zero_plan.cpp", "zero_capi.cpp", "zero_launch.cu", "zero_kernels_fp16.cu",
           "zero_kernels_bf16.cu", "zero_noalloc.cu", "zero_cpu_adam.cpp"]
# extra host-compiler flags per source: the host AdamW loop is vectorised at
# -O3; -fno-math-errno lets sqrtf be the plain instruction (results unchanged)
EXTRA = {"zero_cpu_adam.cpp": ["-Xcompiler", "-O3,-fno-math-errno"]}
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# IEEE division and square root, no flush-to-zero, no FMA contraction of the
# explicitly rounded arithmetic (the kernels use __f*_rn intrinsics anyway).
CUDA_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-prec-div=true", "-prec-sqrt=true",
              "-ftz=false", "-fmad=false", "-Xcompiler", "-fPIC,-O2,-ffp-contract=off",
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libzero.so")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "zero.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def up_to_date() -> bool:
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime()


def build(force: bool = False, verbose: bool = False, extra: list | None = None) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    extra = list(extra or [])

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src + ".o")
        cmd = [cc, *ARCH, *CUDA_FLAGS, *EXTRA.get(src, []), *extra, "-I", INCLUDE, "-I", CSRC, "-c",
               os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
        if verbose and (res.stdout or res.stderr):
            sys.stderr.write(res.stdout + res.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-Xcompiler", "-fPIC"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                extra=["-Xptxas", "-v"] if "--ptxas" in sys.argv else None))
