"""Builds libdetattn.so in-tree from csrc/ with nvcc for sm_103a.

Each translation unit is compiled in its own nvcc process (in parallel), then
the objects are linked into ``_build/libdetattn.so``.  A rebuild happens only
when a source or header is newer than the library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libdetattn.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
SOURCES = ["attn_fwd.cu", "attn_bwd.cu", "attn_dq_ds.cu", "embed_grad.cu", "layer_ops.cu",
           "detattn_host.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdetattn")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)
             if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "detattn.h"))
    files.append(os.path.abspath(__file__))
    return files


def resource_report_path(src: str) -> str:
    """ptxas's resource report (registers, spills, shared memory per kernel)
    of one translation unit, kept from the last build."""
    return os.path.join(BUILD, src.replace(".cu", ".ptxas.txt"))


def up_to_date() -> bool:
    if not os.path.exists(LIB) or not all(os.path.exists(resource_report_path(s)) for s in SOURCES):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    tag = str(os.getpid())

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", f".{tag}.o"))
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-Xptxas", "-v", "-I", INCLUDE, "-c",
               os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        report = resource_report_path(src)
        with open(report + f".tmp{tag}", "w") as f:
            f.write(r.stdout + r.stderr)
        os.replace(report + f".tmp{tag}", report)
        return obj

    objs = [os.path.join(BUILD, src.replace(".cu", f".{tag}.o")) for src in SOURCES]
    try:
        with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
            list(ex.map(compile_one, SOURCES))
        tmp = LIB + f".tmp{tag}"
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    finally:
        # This build's objects go whether it succeeded or not.
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
