"""Builds the CUDA library ``lib/libnm.so`` from ``csrc/*.cu`` with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked
into one shared object with the CUDA runtime linked statically (the library
loads on a host without a GPU driver; CUDA is only touched on the first call
that launches work).  Run ``python -m structured_sparse_gemm_nm_gb300.build``.
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
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libnm.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC,-O2",
              "-I", os.path.join(ROOT, "include")]


def nvcc_path() -> str:
    p = shutil.which("nvcc")
    if p:
        return p
    cand = "/usr/local/cuda/bin/nvcc"
    if os.path.exists(cand):
        return cand
    raise RuntimeError("nvcc not found")


def _compile(src: str, obj: str, extra) -> str:
    cmd = [nvcc_path(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    return r.stderr


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(LIBDIR, exist_ok=True)
    objdir = os.path.join(LIBDIR, "obj")
    os.makedirs(objdir, exist_ok=True)
    srcs = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    jobs = []
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        for f in srcs:
            jobs.append((f, ex.submit(_compile, os.path.join(CSRC, f), os.path.join(objdir, f + ".o"), extra)))
        for f, j in jobs:
            log = j.result()
            if verbose and log:
                print(f"--- {f}\n{log}", file=sys.stderr)
    objs = [os.path.join(objdir, f + ".o") for f in srcs]
    tmp = LIB + ".tmp"
    cmd = [nvcc_path(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv))
