"""Builds the sm_103a shared library libattn_gb300.so in-tree with nvcc.

Each .cu file is compiled as its own translation unit, in parallel, then linked into one
shared library under self_attention_gb300/_build/.  The CUDA runtime is linked statically;
the driver is reached through cudaGetDriverEntryPointByVersion, so no -lcuda is needed.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libattn_gb300.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)

SOURCES = ["attn_api.cu", "attn_fwd.cu", "attn_bwd.cu", "vector_add.cu", "proj.cu", "unfused.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libattn_gb300")
    return cand


def _inputs_newest() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "attn.h"),
                                                                    os.path.abspath(__file__)]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile (if stale) and return the path of libattn_gb300.so."""
    if not force and os.path.exists(LIB_PATH) and os.path.getmtime(LIB_PATH) >= _inputs_newest():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    tool = nvcc()
    tag = f"{os.getpid()}"

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, src.replace(".cu", f".{tag}.o"))
        cmd = [tool, *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.append("-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [o for o, _ in results]
    tmp = LIB_PATH + f".{tag}.tmp"
    r = subprocess.run([tool, *ARCH, "-shared", "-o", tmp, *objs, "-ldl"], capture_output=True, text=True)
    for o in objs:
        os.remove(o)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    if verbose:
        for _, log in results:
            print(log)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force=True, verbose=True))
