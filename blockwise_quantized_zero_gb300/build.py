"""Build libzq.so (the CUDA library behind include/zq.h) in-tree for sm_103a.

Each launch unit in csrc/ is compiled by its own nvcc process (in parallel),
then the objects are linked into ``blockwise_quantized_zero_gb300/libzq.so``
against the shared CUDA runtime. Run ``python -m blockwise_quantized_zero_gb300.build``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libzq.so")

UNITS = ["zq_api.cu", "zq_quantize.cu", "zq_dequantize.cu", "zq_reduce.cu", "zq_fp8.cu",
         "zq_interleave.cu", "zq_reduce_few.cu", "zq_gemm.cu", "zq_quantize_multi.cu"]
HEADERS = ["zq_device.cuh", "zq_kernels.cuh", "zq_host.h", "zq_reduce_launch.h", "zq_tc.cuh",
           "zq_gemm.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# IEEE binary32 everywhere: no FMA contraction (fused forms are written
# explicitly where they are exact), IEEE division and square root, no FTZ.
NVCC_FLAGS = ARCH + [
    "-O3", "-lineinfo", "-std=c++17", "--fmad=false", "-prec-div=true", "-prec-sqrt=true",
    "-ftz=false", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC,
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", shutil.which("nvcc")):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libzq")


def _cuda_lib_dir(nvcc: str) -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "lib64")


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "zq.h"),
                                                                os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False) -> str:
    """Compile and link libzq.so; returns its path. Raises on a compiler error."""
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    flags = NVCC_FLAGS + (["-Xptxas", "-v"] if ptxas_info else [])

    def compile_unit(unit):
        src = os.path.join(CSRC, unit)
        obj = os.path.join(BUILD, unit.replace(".cu", ".o"))
        if not force and not ptxas_info and not _stale(obj, src):
            return obj, ""
        cmd = [nvcc, *flags, "-c", src, "-o", obj]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"nvcc failed on {unit}:\n{p.stdout}\n{p.stderr}")
        return obj, p.stdout + p.stderr

    with cf.ThreadPoolExecutor(len(UNITS)) as ex:
        results = list(ex.map(compile_unit, UNITS))
    if verbose or ptxas_info:
        for _, log in results:
            if log:
                print(log)
    objs = [o for o, _ in results]
    if force or not os.path.exists(LIB) or any(os.path.getmtime(o) > os.path.getmtime(LIB) for o in objs):
        libdir = _cuda_lib_dir(nvcc)
        tmp = LIB + ".tmp"
        cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
               "-Xlinker", "-rpath=" + libdir]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"link failed:\n{p.stdout}\n{p.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True, ptxas_info="-v" in sys.argv, force="-f" in sys.argv))
