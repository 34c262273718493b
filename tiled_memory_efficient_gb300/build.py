"""Builds the CUDA library libattn.so in-tree with nvcc (sm_103a only).

    python -m tiled_memory_efficient_gb300.build [--force]

Each .cu file compiles in parallel to an object file under _build/, then one
link step produces _build/libattn.so against the shared CUDA runtime.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libattn.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

SOURCES = ["abi.cu", "attn_fwd.cu", "attn_bwd.cu", "bwd_noalloc.cu", "splitkv.cu", "ffn.cu",
           "vconv.cu"]
HEADERS = ["ptx.cuh", "attn_internal.h", "bias.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-v"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files += [os.path.join(INCLUDE, h) for h in ("attn.h", "ffn.h")]
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime():
        return LIB
    cc = nvcc()
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        log = open(os.path.join(BUILD, src.replace(".cu", ".log")), "w")
        cmd = [cc, *ARCH, *FLAGS, "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        procs.append((src, subprocess.Popen(cmd, stdout=log, stderr=subprocess.STDOUT), log))
        objs.append(obj)
    failed = []
    for src, pr, log in procs:
        rc = pr.wait()
        log.close()
        if rc != 0:
            failed.append(src)
    if failed:
        msgs = []
        for src in failed:
            with open(os.path.join(BUILD, src.replace(".cu", ".log"))) as f:
                msgs.append(f"--- {src}\n" + f.read()[-6000:])
        raise RuntimeError("nvcc failed:\n" + "\n".join(msgs))
    if verbose:
        for src in SOURCES:
            with open(os.path.join(BUILD, src.replace(".cu", ".log"))) as f:
                print(f.read())
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([cc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
