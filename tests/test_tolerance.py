"""The attention error bound (tests/tolerance.py) against the arithmetic it
claims to cover, on the CPU.

The kernels' arithmetic is emulated in numpy step by step (fp32 scores from
bf16 inputs, p in fp32 against a reference that may lag the maximum by up to
2^8, p rounded to bf16 for the numerator, the unrounded p summed for the
denominator, the bf16 output rounded to nearest even) and compared with the
exact value in double: every element must sit inside the bound, and the P
term must be needed (without it the emulation leaves the bound on peaked
rows) — so the bound is neither too tight for a correct kernel nor vacuous.
"""
from __future__ import annotations

import numpy as np
import pytest

from tests import tolerance as tol


def to_bf16(x):
    """Round float32 values to bf16 (nearest, ties to even); returns float32."""
    b = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (b.astype(np.uint32) << 16).view(np.float32)


def emulate(q, k, v, scale, lag):
    """One query row: fp32 scores, p = 2^(s*scale*log2e - m_ref) with
    m_ref = max - lag, bf16 p in the numerator, fp32 p in the denominator."""
    s = (k.astype(np.float32) @ q.astype(np.float32)).astype(np.float32)
    x = (s * np.float32(scale * np.log2(np.e))).astype(np.float32)
    m_ref = np.float32(x.max() - lag)
    p = np.exp2((x - m_ref).astype(np.float32)).astype(np.float32)
    l = np.float32(p.sum(dtype=np.float32))
    num = (to_bf16(p)[None, :] @ v.astype(np.float32)).astype(np.float32)[0]
    return to_bf16(num / l)


def exact(q, k, v, scale):
    s = (k.astype(np.float64) @ q.astype(np.float64)) * scale
    w = np.exp(s - s.max())
    w /= w.sum()
    return w @ v.astype(np.float64), w @ np.abs(v.astype(np.float64))


@pytest.mark.parametrize("n,peak", [(1, 1.0), (2, 1.0), (5, 4.0), (17, 6.0), (64, 1.0), (700, 1.0), (3000, 2.0)])
def test_bound_covers_the_kernel_arithmetic(n, peak):
    rng = np.random.default_rng(n)
    d = 128
    scale = 1 / np.sqrt(d)
    worst = 0.0
    for trial in range(40):
        q = to_bf16(rng.standard_normal(d) * peak)
        k = to_bf16(rng.standard_normal((n, d)) * peak)
        v = to_bf16(rng.standard_normal((n, d)) * (1 + 2 * (trial % 3)))
        ref, a_abs = exact(q, k, v, scale)
        for lag in (0.0, 3.7, 7.9):
            got = emulate(q, k, v, scale, lag)
            err = np.abs(got - ref)
            b = tol.bound(ref, a_abs)
            assert (err <= b).all(), (n, trial, lag, float((err / b).max()))
            worst = max(worst, float((err / b).max()))
    if n > 1:   # (one key: o = v exactly)
        assert worst > 0.05   # the bound is not orders of magnitude above what happens


def test_p_rounding_term_is_needed():
    """Without u_P * A (flat 1e-2 and output rounding only) peaked rows with
    large values leave the bound: the term is part of what the arithmetic
    forces, not slack."""
    rng = np.random.default_rng(7)
    d, scale = 128, 1 / np.sqrt(128)
    outside = 0
    for trial in range(400):
        n = int(rng.integers(2, 6))
        q = to_bf16(rng.standard_normal(d) * 3)
        k = to_bf16(rng.standard_normal((n, d)) * 3)
        v = to_bf16(rng.standard_normal((n, d)) * 6)
        ref, a_abs = exact(q, k, v, scale)
        got = emulate(q, k, v, scale, 5.3)
        err = np.abs(got - ref)
        assert (err <= tol.bound(ref, a_abs)).all()
        no_p = np.maximum(tol.MAX_ABS, tol.bf16_ulp(np.abs(ref)) / 2)
        outside += int((err > no_p).sum())
    assert outside > 0


def test_bound_values():
    # flat 1e-2 for small outputs; half an ulp plus the P term above
    assert tol.bound(np.array([0.3]), np.array([0.8]))[0] == pytest.approx(1e-2)
    b = tol.bound(np.array([3.0]), np.array([3.0]))[0]
    e = 2 ** -8 * 3 + tol.FP32_SLACK * 6
    assert b == pytest.approx(e + 2 ** -7, rel=1e-12)   # ulp in [2, 4) is 2^-6
