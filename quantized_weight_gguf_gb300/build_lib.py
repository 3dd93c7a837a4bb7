"""Build libqmm.so in-tree with nvcc for sm_103a (one -gencode, translation
units compiled in parallel, then linked). Usable as ``python -m
quantized_weight_gguf_gb300.build_lib`` or through ``build()``."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqmm.so")
# the tensor-core kernel instances come first: they take longest to compile
SOURCES = ["qmm_mma_inst_q4k.cu", "qmm_mma_inst_16.cu", "qmm_mma_inst_q.cu", "qmm_mma_inst_aff.cu",
           "qmm_mma_inst_grp.cu",
           "qmm_api.cu", "qmm_gemv.cu", "qmm_mma.cu", "qmm_dequant.cu", "qmm_noalloc.cu",
           "qmm_back_input.cu"]
GENCODE = "arch=compute_103a,code=sm_103a"


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libqmm")


def _flags():
    return ["-gencode", GENCODE, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
            "-I", os.path.join(ROOT, "include"), "--expt-relaxed-constexpr"]


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    t = os.path.getmtime(obj)
    deps = [src] + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(ROOT, "include", "qmm.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    nvcc = nvcc_path()
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(BUILD, src.replace(".cu", ".o"))
        if force or _stale(o, s):
            jobs.append((s, o))

    def compile_one(so):
        s, o = so
        cmd = [nvcc, *_flags(), "-c", s, "-o", o + ".tmp"]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(s)}:\n{r.stdout}\n{r.stderr}")
        os.replace(o + ".tmp", o)
        return r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        for log in ex.map(compile_one, jobs):
            if verbose and log:
                sys.stderr.write(log)
    objs = [os.path.join(BUILD, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or not os.path.exists(LIB):
        tmp = LIB + f".{os.getpid()}.tmp"
        cmd = [nvcc, "-gencode", GENCODE, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs,
               "-lcudart"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
