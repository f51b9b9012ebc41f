"""Builds the CUDA library in-tree: block_wise_fp8_gb300/_build/libfp8bq.so.

One nvcc process per translation unit, run in parallel, for sm_103a only; the
objects are linked into a shared library with the CUDA runtime linked
statically, so loading it needs no GPU (only calling it does).
"""
from __future__ import annotations

import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libfp8bq.so")
# the debug build: the same sources with FP8BQ_DEBUG_CHECKS (device-side bounds
# checks on the GEMM epilogues' writes, reported as FP8BQ_ERR_BOUNDS)
OUT_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(OUT_DEBUG, "libfp8bq.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

SOURCES = ["fp8bq_api.cu", "quant.cu", "gemm_launch.cu", "gemm_block.cu",
           "gemm_tensor.cu", "gemm_mx.cu", "gemm_channel.cu",
           "norm_quant.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps() -> list[str]:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
             if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "fp8bq.h"))
    return files


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    out, lib = (OUT_DEBUG, LIB_DEBUG) if debug else (OUT, LIB)
    if not force and up_to_date(lib):
        return lib
    os.makedirs(out, exist_ok=True)
    nvcc = _nvcc()
    procs = []
    objs = []
    extra = ["-DFP8BQ_DEBUG_CHECKS"] if debug else []
    for src in SOURCES:
        obj = os.path.join(out, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                            stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode:
            print(f"--- nvcc {src}\n{out}", flush=True)
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib + f".tmp{os.getpid()}"
    link = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lpthread", "-ldl", "-lrt"]
    subprocess.run(link, check=True)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                debug="--debug" in sys.argv))
