"""Prefix hash -> bf16 values, and the synthetic next-token model.

Definitions (numpy, CPU).  ``synth/csrc/synth_gen.cu`` restates the same
integer definitions for the GPU so that bench-sized inputs can be made on the
device; a test checks the two agree bit for bit.

* ``mix64`` is the output finaliser of splitmix64 (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014), with the
  constants published there.
* Prefix hash of a token sequence x_0..x_{n-1}:
  ``h_{-1} = mix64(seed)``, ``h_i = mix64(h_{i-1} XOR mix64((x_i + 1) * GAMMA))``.
  Every value of token i is a function of ``h_i`` alone, so two requests with
  the same prefix get the same K/V, which is what makes cache reuse exactly
  checkable.
* Element (layer, kind, head, dim) of token i: three splitmix64 outputs
  ``w_j = mix64(h_i + (3*key + j + 1) * GAMMA)``, ``key = ((layer*4 + kind)*256
  + head)*1024 + dim``; their twelve 16-bit fields u_q are summed and
  ``v = (sum - 6*65536) / 65536`` (Irwin-Hall with 12 terms: mean 0, variance 1
  up to the 2^-16 quantisation).  ``v`` is exact in float32 and is rounded to
  bf16 with round-to-nearest-even.
* Decode model: the token that follows prefix hash h is
  ``mix64(h XOR TOKEN_SALT) mod vocab``.
"""
from __future__ import annotations

import numpy as np

MASK64 = (1 << 64) - 1
GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
TOKEN_SALT = 0xD1B54A32D192ED03

KIND_K, KIND_V, KIND_Q = 0, 1, 2

_U = np.uint64


def mix64(x):
    """splitmix64 finaliser on a Python int or a uint64 array (wrapping)."""
    if isinstance(x, (int, np.integer)) and not isinstance(x, np.ndarray):
        z = int(x) & MASK64
        z = ((z ^ (z >> 30)) * _M1) & MASK64
        z = ((z ^ (z >> 27)) * _M2) & MASK64
        return z ^ (z >> 31)
    z = np.asarray(x, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> _U(30))) * _U(_M1)
        z = (z ^ (z >> _U(27))) * _U(_M2)
    return z ^ (z >> _U(31))


def root_hash(seed: int) -> int:
    """h_{-1}: the hash state before the first token of every sequence."""
    return mix64(seed)


def _token_mix(tokens: np.ndarray) -> np.ndarray:
    t = np.asarray(tokens, dtype=np.int64).astype(np.uint64)
    with np.errstate(over="ignore"):
        return mix64((t + _U(1)) * _U(GAMMA))


def prefix_hashes_from(h_prev: int, tokens) -> np.ndarray:
    """Continue a prefix-hash chain from state ``h_prev`` over ``tokens``."""
    tm = [int(v) for v in _token_mix(np.asarray(tokens).reshape(-1))]
    out = np.empty(len(tm), dtype=np.uint64)
    h = int(h_prev) & MASK64
    for i, t in enumerate(tm):
        h = mix64(h ^ t)
        out[i] = h
    return out


def prefix_hashes(tokens, seed: int) -> np.ndarray:
    """h_0..h_{n-1} of one sequence."""
    return prefix_hashes_from(root_hash(seed), tokens)


def prefix_hashes_rows(tokens2d: np.ndarray, h_prev: np.ndarray) -> np.ndarray:
    """Vectorised over rows: continue each row's chain from ``h_prev[row]``."""
    tokens2d = np.asarray(tokens2d)
    tm = _token_mix(tokens2d)
    out = np.empty(tokens2d.shape, dtype=np.uint64)
    h = np.asarray(h_prev, dtype=np.uint64).copy()
    for i in range(tokens2d.shape[1]):
        h = mix64(h ^ tm[:, i])
        out[:, i] = h
    return out


def _f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round-to-nearest-even float32 -> bf16 bit pattern (finite inputs)."""
    b = np.asarray(f, dtype=np.float32).view(np.uint32).astype(np.uint64)
    b = (b + _U(0x7FFF) + ((b >> _U(16)) & _U(1))) >> _U(16)
    return b.astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def gen_values(hashes, kind: int, heads: int, dims: int, layer: int = 0,
               head0: int = 0, chunk: int = 4096) -> np.ndarray:
    """bf16 bit patterns, shape [n, heads, dims], of the given kind.

    ``head0`` offsets the head index (to draw a subset of heads).
    """
    h = np.asarray(hashes, dtype=np.uint64).reshape(-1)
    n = h.shape[0]
    out = np.empty((n, heads, dims), dtype=np.uint16)
    head = np.arange(head0, head0 + heads, dtype=np.uint64)[:, None]
    dim = np.arange(dims, dtype=np.uint64)[None, :]
    key = ((_U(layer * 4 + kind) * _U(256) + head) * _U(1024) + dim)  # [heads, dims]
    with np.errstate(over="ignore"):
        offs = [(key * _U(3) + _U(j + 1)) * _U(GAMMA) for j in range(3)]
    for s in range(0, n, chunk):
        hc = h[s:s + chunk][:, None, None]
        acc = np.zeros((hc.shape[0], heads, dims), dtype=np.int64)
        for j in range(3):
            with np.errstate(over="ignore"):
                w = mix64(hc + offs[j][None])
            for q in range(4):
                acc += ((w >> _U(16 * q)) & _U(0xFFFF)).astype(np.int64)
        v = (acc - 6 * 65536).astype(np.float32) / np.float32(65536.0)
        out[s:s + chunk] = _f32_to_bf16_bits(v)
    return out


def gen_token(h: int, vocab: int) -> int:
    """The synthetic model's next token after a prefix with hash ``h``."""
    return mix64((int(h) ^ TOKEN_SALT) & MASK64) % vocab


def gen_tokens(hashes: np.ndarray, vocab: int) -> np.ndarray:
    """Vectorised ``gen_token``."""
    return (mix64(np.asarray(hashes, dtype=np.uint64) ^ _U(TOKEN_SALT)) % _U(vocab)).astype(np.int32)
