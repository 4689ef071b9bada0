"""Oracle of the FP8 (E4M3) KV pool: test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module; it shares no code with the product library.

The SGLang engineering article on DeepSeek support, section 1: the KV cache is
quantised to FP8, and block-wise FP8 stores activations as E4M3 with one
dynamic scale per token per 128-channel group.  Reading for the KV pool: one
fp32 scale per (token, KV head) row of 128 channels, scale = amax / 448 (448
being E4M3's largest finite value), code_i = E4M3(x_i / scale); both quotients
are fp32 divisions rounded to nearest, and E4M3 rounding is to the nearest
representable value, ties to the even code, saturating at +-448.  An all-zero
row has scale 0 and zero codes.  A row's values are code * scale.

E4M3 (the OCP 8-bit floating point format): sign, 4 exponent bits (bias 7),
3 mantissa bits; exponent 0 holds subnormals m * 2^-9; 0x7F / 0xFF are NaN;
no infinities.

Attention over an FP8 pool is the plain definition (two-pass softmax in
double) applied to the dequantised K/V and the bf16 queries.

Parity status: pinned by tests/test_fp8_oracle.py -- the format's published
values (largest finite 448, smallest normal 2^-6, smallest subnormal 2^-9,
1.0 = 0x38), brute-force nearest-value search over all finite codes for the
rounding, the quantisation error bound, and equality with the separately
pinned bf16 attention oracle on inputs that quantise exactly.
"""
from __future__ import annotations

import numpy as np

E4M3_MAX = 448.0


def decode_table() -> np.ndarray:
    """Value of every code 0..255 (NaN for 0x7F and 0xFF), float64."""
    out = np.empty(256, np.float64)
    for c in range(256):
        sign = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 7
        if e == 15 and m == 7:
            out[c] = np.nan
        elif e == 0:
            out[c] = sign * m * 2.0 ** -9
        else:
            out[c] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return out


def encode(y) -> np.ndarray:
    """Nearest E4M3 code of each value (float64 array), ties to even,
    saturating at +-448.  A value that rounds to zero keeps its sign."""
    y = np.asarray(y, np.float64)
    a = np.abs(y)
    codes = np.zeros(y.shape, np.uint8)
    big = a >= E4M3_MAX
    nz = (a > 0) & ~big
    e = np.full(y.shape, -6.0)
    e[nz] = np.maximum(np.floor(np.log2(a[nz])), -6.0)
    quantum = 2.0 ** (e - 3)
    k = np.rint(np.where(nz, a / quantum, 0.0))   # multiples of the quantum, ties to even
    v = k * quantum
    mag = np.zeros(y.shape, np.int64)
    sub = nz & (v < 2.0 ** -6)
    mag[sub] = (v[sub] / 2.0 ** -9).astype(np.int64)
    nrm = nz & (v >= 2.0 ** -6)
    ev = np.floor(np.log2(np.where(nrm, v, 1.0)))
    mant = np.where(nrm, v / 2.0 ** ev * 8.0 - 8.0, 0.0)
    mag[nrm] = ((ev[nrm].astype(np.int64) + 7) << 3) | mant[nrm].astype(np.int64)
    mag[big] = 0x7E
    codes[:] = mag.astype(np.uint8)
    codes |= np.where(np.signbit(y), 0x80, 0).astype(np.uint8)
    return codes


def quantize_rows(x_bits) -> tuple:
    """Rows of bf16 bits [..., 128] -> (codes uint8 [..., 128], scales float32 [...])."""
    x = (np.asarray(x_bits, np.uint16).astype(np.uint32) << 16).view(np.float32)
    amax = np.max(np.abs(x), axis=-1)
    scale = (amax / np.float32(E4M3_MAX)).astype(np.float32)   # fp32 division, nearest
    safe = np.where(scale > 0, scale, np.float32(1.0)).astype(np.float32)
    y = (x / safe[..., None]).astype(np.float32)                # fp32 division, nearest
    codes = encode(y.astype(np.float64))
    codes[scale == 0] = 0
    return codes, scale


def dequantize(codes, scales) -> np.ndarray:
    return decode_table()[np.asarray(codes, np.int64)] * np.asarray(scales, np.float64)[..., None]


def attention(q_bits, k, v, kv_off, ctx, q_heads, kv_heads, scale):
    """Exact attention in double.  q_bits: bf16 bits [rows, Hq, D]; k, v:
    dequantised values [tokens, Hkv, D] (float64).  Row r sees tokens
    kv_off[r] .. kv_off[r]+ctx[r]-1.  Returns (out [rows, Hq, D], lse [rows, Hq])."""
    q = (np.asarray(q_bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    rows, D = q.shape[0], q.shape[2]
    g = q_heads // kv_heads
    out = np.empty((rows, q_heads, D), np.float64)
    lse = np.empty((rows, q_heads), np.float64)
    for r in range(rows):
        a, n = int(kv_off[r]), int(ctx[r])
        for h in range(q_heads):
            kh, vh = k[a:a + n, h // g], v[a:a + n, h // g]
            s = (kh @ q[r, h]) * scale
            m = s.max()
            p = np.exp(s - m)
            l = p.sum()
            out[r, h] = (p @ vh) / l
            lse[r, h] = m + np.log(l)
    return out, lse
