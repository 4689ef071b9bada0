"""Pins of the FP8 (E4M3) KV-pool oracle against the format's published
values, brute force and the separately pinned bf16 attention oracle (CPU)."""
from __future__ import annotations

import numpy as np
import pytest

import oracle
from oracle import fp8_oracle as f8


def test_e4m3_published_values():
    t = f8.decode_table()
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0           # largest finite
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])          # the only NaNs, no infinities
    assert t[0x08] == 2.0 ** -6 and t[0x01] == 2.0 ** -9    # smallest normal, smallest subnormal
    assert t[0x38] == 1.0 and t[0xC0] == -2.0 and t[0x00] == 0.0
    finite = t[~np.isnan(t)]
    assert len(finite) == 254 and len(np.unique(finite)) == 253   # +0 and -0
    pos = t[:0x7F]
    assert (np.diff(pos) > 0).all()                          # codes ordered by value


def test_encode_is_nearest_with_ties_to_even_brute_force():
    t = f8.decode_table()
    codes = np.arange(0x7F)                                  # non-negative finite codes
    vals = t[codes]
    rng = np.random.default_rng(0)
    y = np.concatenate([rng.uniform(0, 460, 4000), rng.uniform(0, 2.0 ** -5, 4000),
                        (vals[:-1] + vals[1:]) / 2,          # every tie
                        vals, [448.0, 449.0, 464.0, 1e6]])
    got = f8.encode(y)
    for yi, c in zip(y, got):
        d = np.abs(vals - min(yi, 448.0))
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else best[best % 2 == 0][0]   # tie: even code
        assert c == want, (yi, c, want)
    neg = f8.encode(-y)
    assert (neg == (got | 0x80)).all()                       # sign symmetric


def test_quantize_rows_error_bound_and_amax():
    rng = np.random.default_rng(1)
    x = rng.standard_normal((64, 128)).astype(np.float32) * rng.uniform(1e-3, 50, (64, 1)).astype(np.float32)
    xb = (x.view(np.uint32) >> 16).astype(np.uint16)        # truncate to bf16 bits
    xv = (xb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    codes, scale = f8.quantize_rows(xb)
    deq = f8.dequantize(codes, scale)
    amax = np.abs(xv).max(axis=1)
    # the largest element lands on +-448 * scale, within one fp32 rounding
    assert np.allclose(np.abs(deq).max(axis=1), amax, rtol=1e-6)
    # normal range: half an E4M3 step (2^-4 relative) plus the quotient's rounding
    big = np.abs(xv) >= scale[:, None] * 2.0 ** -6
    rel = np.abs(deq - xv)[big] / np.abs(xv)[big]
    assert rel.max() <= 2.0 ** -4 * (1 + 1e-6)
    # subnormal range: absolute error at most half of 2^-9 * scale
    small = ~big
    assert (np.abs(deq - xv)[small] <= (2.0 ** -10 * scale[:, None] * (1 + 1e-6)).repeat(128, 1)[small]).all()
    # an all-zero row: scale 0, codes 0
    c0, s0 = f8.quantize_rows(np.zeros((1, 128), np.uint16))
    assert s0[0] == 0 and (c0 == 0).all()


def test_fp8_attention_equals_bf16_oracle_on_exact_inputs():
    """Inputs whose quantisation is exact (E4M3 values times 1/8, row amax
    56 = 448/8): the FP8 oracle equals the bf16 attention oracle."""
    rng = np.random.default_rng(2)
    t = f8.decode_table()
    finite = np.flatnonzero(~np.isnan(t) & (np.abs(t) <= 448))
    T, Hkv, Hq, D = 40, 2, 8, 128

    def rows():
        c = rng.choice(finite, (T, Hkv, D))
        c[:, :, 0] = 0x7E                                      # amax = 448 codes -> scale 1/8
        return t[c] / 8.0

    kv = [rows(), rows()]
    bf = [((v.astype(np.float32).view(np.uint32)) >> 16).astype(np.uint16) for v in kv]
    assert all(((b.astype(np.uint32) << 16).view(np.float32) == v).all() for b, v in zip(bf, kv))
    q = (rng.standard_normal((3, Hq, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    qk = [f8.quantize_rows(b) for b in bf]
    deq = [f8.dequantize(c, s) for c, s in qk]
    assert all(np.array_equal(d, v) for d, v in zip(deq, kv))
    off, ctx = np.array([0, 5, 0]), np.array([40, 20, 1])
    o1, l1 = f8.attention(q, deq[0], deq[1], off, ctx, Hq, Hkv, 1 / np.sqrt(D))
    o2, l2 = oracle.attention(q, bf[0], bf[1], off, ctx, Hq, Hkv, D, D, 1 / np.sqrt(D))
    assert np.abs(o1 - o2).max() <= 1e-12 and np.abs(l1 - l2).max() <= 1e-12


@pytest.mark.parametrize("n", [1, 7])
def test_fp8_attention_closed_forms(n):
    """One key: the output is that key's value; equal keys: the mean."""
    rng = np.random.default_rng(n)
    D, Hq, Hkv = 128, 4, 1
    v = rng.standard_normal((n, Hkv, D))
    k = np.repeat(rng.standard_normal((1, Hkv, D)), n, 0)
    q = (rng.standard_normal((1, Hq, D)).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    o, _ = f8.attention(q, k, v, np.array([0]), np.array([n]), Hq, Hkv, 0.1)
    assert np.allclose(o[0], v.mean(0)[0][None, :], atol=1e-12)
