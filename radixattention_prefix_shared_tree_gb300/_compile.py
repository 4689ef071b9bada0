"""Build the C-ABI library ``_build/libradixattn.so`` in-tree with nvcc (sm_103a).

Translation units compile in parallel; the host tree is plain C++ (g++), the
kernels are CUDA for ``arch=compute_103a,code=sm_103a``.  cudart is linked
statically so the library does not depend on which libcudart the process
already loaded.
"""
from __future__ import annotations

import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libradixattn.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

CU_SOURCES = ["kv_store.cu", "attn_decode.cu", "attn_decode_mla.cu", "attn_extend.cu", "runtime.cu"]
CPP_SOURCES = ["radix_cache.cpp", "block_cache.cpp"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    p = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(p):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return p


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "radixattn.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(f) <= t for f in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    nv = nvcc()
    jobs = []
    objs = []
    for src in CU_SOURCES:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nv] + ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                             "-c", os.path.join(CSRC, src), "-o", obj]
        jobs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    for src in CPP_SOURCES:
        obj = os.path.join(BUILD, src.replace(".cpp", ".o"))
        cmd = ["g++", "-O3", "-std=c++17", "-fPIC", "-I", INCLUDE, "-c", os.path.join(CSRC, src), "-o", obj]
        jobs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
        objs.append(obj)
    failed = []
    for src, pr in jobs:
        out, _ = pr.communicate()
        if verbose or pr.returncode:
            print(out.decode(errors="replace"))
        if pr.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError(f"compilation failed: {failed}")
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nv] + ARCH + ["-shared", "-o", tmp] + objs + ["-lstdc++"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))
