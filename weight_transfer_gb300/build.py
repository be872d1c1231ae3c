"""Build libfp8q.so in place: one nvcc object per .cu, compiled in parallel,
linked into a shared library next to this file.

Flags: sm_103a only, -O3, line info, no fast-math, explicitly no
flush-to-zero, IEEE division and square root, and -fmad=false so that no
multiply-add pair is contracted into an FMA behind the source's back.
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
LIB = os.path.join(HERE, "libfp8q.so")

SOURCES = ["api.cu", "quantize.cu", "reduce.cu", "ring_hop.cu", "mxfp8.cu", "mxfp8_receive.cu", "ring_allreduce.cu", "tensorwise.cu", "pack.cu", "selftest.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-ftz=false", "-prec-div=true", "-prec-sqrt=true",
                  "-fmad=false", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libfp8q.so")
    return path


def _inputs():
    hdrs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    return [os.path.join(CSRC, s) for s in SOURCES], hdrs + [os.path.join(INCLUDE, "fp8q.h")]


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    srcs, hdrs = _inputs()
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(p) <= t for p in srcs + hdrs + [__file__])


def nvtx_requested() -> bool:
    """FP8Q_NVTX=1 in the environment compiles the NVTX ranges in (off by default)."""
    return os.environ.get("FP8Q_NVTX", "0") not in ("", "0")


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    stamp = os.path.join(BUILD, "nvtx" if nvtx_requested() else "plain")
    if not force and up_to_date() and os.path.exists(stamp):
        return LIB
    if os.path.isdir(BUILD):
        for f in ("nvtx", "plain"):
            if os.path.exists(os.path.join(BUILD, f)):
                os.remove(os.path.join(BUILD, f))
    os.makedirs(BUILD, exist_ok=True)
    cc = nvcc()
    srcs, _ = _inputs()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if nvtx_requested():
        extra += ["-DFP8Q_NVTX=1"]

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src).replace(".cu", ".o"))
        cmd = [cc] + NVFLAGS + extra + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        results = list(ex.map(compile_one, srcs))
    if verbose or ptxas_info:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    open(stamp, "w").close()
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas-info" in sys.argv)
    print(LIB)
