"""Builds libfsdpstate.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in its own nvcc process, in parallel; the shared
library lands in ``fsdp_sharded_state_gb300/_build/``.  No cmake, no torch
extension machinery: the library is plain C ABI.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "_build")
LIB = os.path.join(OUT, "libfsdpstate.so")
SOURCES = ["api.cu", "kernels.cu", "layout.cpp", "noalloc.cu", "rows.cu", "staged.cu", "allgather.cu", "staged_rows.cu",
           "clip_coop.cu", "claims.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# IEEE division and square root, no flush-to-zero, no implicit fma contraction:
# the kernels spell out every fma they want.
NVFLAGS = ["-O3", "-std=c++17", "-lineinfo", "--fmad=false", "-prec-div=true", "-prec-sqrt=true",
           "-ftz=false", "-Xcompiler", "-fPIC,-O2,-fno-fast-math", "-Xptxas", "-warn-spills"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfsdpstate")


def _newer(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    os.makedirs(OUT, exist_ok=True)
    cc = nvcc()
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".hpp"))]
    headers.append(os.path.join(HERE, "..", "include", "fsdp_state.h"))
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OUT, src + ".o")
        objs.append(o)
        if force or ptxas_info or _newer(o, [s, *headers, __file__]):
            flags = list(NVFLAGS)
            if ptxas_info and src.endswith(".cu"):
                flags += ["-Xptxas", "-v"]
            jobs.append([cc, *ARCH, *flags, "-c", s, "-o", o])
    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(lambda c: subprocess.run(c, capture_output=True, text=True), jobs))
    for cmd, r in zip(jobs, results):
        if verbose or ptxas_info:
            print(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        # a front-end diagnostic (e.g. #549-D, a variable read before it is set) fails the
        # build; ptxas's register-spill notes do not
        if "warning #" in r.stdout + r.stderr:
            os.remove(cmd[cmd.index("-o") + 1])
            raise RuntimeError(f"nvcc warned: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if force or _newer(LIB, objs):
        tmp = LIB + f".tmp{os.getpid()}"
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static", "-lrt", "-ldl", "-lpthread"],
                           capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
