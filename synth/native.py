"""ctypes binding of synth/csrc/synth_gen.cu (built to synth/_build/libsynth.so).

Same definitions as synth/hashgen.py, for inputs too large for numpy: a host
prefix-hash scan, the synthetic decode model, and a GPU kernel that writes the
bf16 values of many tokens straight into device memory.
"""
from __future__ import annotations

import ctypes as C
import os
import shutil
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "csrc", "synth_gen.cu")
LIB = os.path.join(HERE, "_build", "libsynth.so")


def build(force: bool = False) -> str:
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call([nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17",
                           "-Xcompiler", "-fPIC", "-shared", "-o", tmp, SRC])
    os.replace(tmp, LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            raise RuntimeError(f"{LIB} is missing: run synth.native.build()")
        L = C.CDLL(LIB)
        VP, I64, I32, U64 = C.c_void_p, C.c_int64, C.c_int32, C.c_uint64
        L.synth_prefix_hashes.argtypes = [VP, I64, U64, VP]
        L.synth_prefix_hashes.restype = None
        L.synth_decode_tokens.argtypes = [U64, I64, I32, VP, VP]
        L.synth_decode_tokens.restype = None
        L.synth_gen_values.argtypes = [VP, I64, I32, I32, I32, I32, I32, VP, I64, VP]
        L.synth_gen_values.restype = C.c_int
        _lib = L
    return _lib


def prefix_hashes_from(h_prev: int, tokens) -> np.ndarray:
    t = np.ascontiguousarray(tokens, dtype=np.int32)
    out = np.empty(len(t), np.uint64)
    if len(t):
        lib().synth_prefix_hashes(t.ctypes.data_as(C.c_void_p), len(t), C.c_uint64(int(h_prev)),
                                  out.ctypes.data_as(C.c_void_p))
    return out


def decode_tokens(h: int, m: int, vocab: int):
    """The synthetic model's next m tokens after a prefix of hash h, and the hashes after each."""
    tok = np.empty(max(m, 1), np.int32)
    hs = np.empty(max(m, 1), np.uint64)
    if m:
        lib().synth_decode_tokens(C.c_uint64(int(h)), m, vocab, tok.ctypes.data_as(C.c_void_p),
                                  hs.ctypes.data_as(C.c_void_p))
    return tok[:m], hs[:m]


def gen_values_gpu(d_hashes, kind: int, heads: int, dims: int, out, layer: int = 0, head0: int = 0,
                   stream=None):
    """Write values for hashes d_hashes [n] (torch int64 on device) into out [n, ...] (bf16/int16 view).

    Row t of ``out`` (stride out.stride(0) elements) receives heads x dims values.
    """
    import torch
    n = d_hashes.numel()
    s = stream if stream is not None else torch.cuda.current_stream()
    st = lib().synth_gen_values(C.c_void_p(d_hashes.data_ptr()), n, layer, kind, heads, dims, head0,
                                C.c_void_p(out.data_ptr()), out.stride(0), C.c_void_p(s.cuda_stream))
    if st != 0:
        raise RuntimeError("synth_gen_values launch failed")
