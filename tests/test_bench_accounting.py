"""The benchmark's accounting on the CPU, each against a count made another
way: a decode step's algorithmic bytes are the union of the K/V rows the
step reads (a shared prefix once) plus indices, Q, O and the stored token;
extend flops are 4·d·Hq per unmasked (query, key) pair of an explicit causal
mask; the clock sampler reads nvidia-smi's lines into a median clock and the
throttle reasons that reject a run."""
from __future__ import annotations

import json
import os
from types import SimpleNamespace

import numpy as np
import pytest

import bench
from radixattention_prefix_shared_tree_gb300.driver import plan_from_rows
from synth.traces import GQA_32_8, GQA_64_8

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _tree_rows():
    """Prompt rows of an agent-style batch: a root shared by all six, two
    branches shared by three each, private tails; slots are distinct ids."""
    nxt = iter(range(10_000))
    take = lambda n: [next(nxt) for _ in range(n)]
    root = take(40)
    branches = [take(17), take(9)]
    rows = []
    for b in range(6):
        rows.append(np.array(root + branches[b // 3] + take(5 + 3 * b), np.int32))
    return rows


def _fake_layout(rows, cascade):
    plan = plan_from_rows(rows) if cascade else dict(n_seg=0)
    B = len(rows)
    lay = SimpleNamespace(L=np.array([len(r) for r in rows], np.int64), batch_size=B,
                          use_cascade=cascade and plan["n_seg"] > 0, private=np.zeros(B, np.int64), segments=[])
    if lay.use_cascade:
        lay.private = plan["private"].astype(np.int64)
        ip, rip = plan["seg_indptr"], plan["seg_row_indptr"]
        lay.segments = [(plan["seg_slots"][ip[k]:ip[k + 1]], plan["seg_rows"][rip[k]:rip[k + 1]])
                        for k in range(plan["n_seg"])]
    return lay


@pytest.mark.parametrize("shape", [GQA_32_8, GQA_64_8])
@pytest.mark.parametrize("t", [0, 7])
def test_decode_bytes_is_the_union_of_rows_read(shape, t):
    rows = _tree_rows()
    B = len(rows)
    # step t: each request reads its prompt rows and its first t + 1 decode
    # rows (new, distinct slots)
    dec = [list(range(20_000 + 1000 * b, 20_000 + 1000 * b + t + 1)) for b in range(B)]
    union = set()
    for r, d in zip(rows, dec):
        union.update(int(x) for x in r)
        union.update(d)
    R = 2 * shape.kv_heads * shape.head_dim_k * 2
    qo = B * shape.q_heads * (shape.head_dim_k + shape.head_dim_v) * 2
    lay = _fake_layout(rows, cascade=True)
    assert lay.use_cascade and len(lay.segments) == 3
    unique, logical = bench.decode_bytes(lay, t, shape)
    assert unique == len(union) * (R + 4) + qo + B * R
    assert logical == sum(len(r) + t + 1 for r in rows) * R
    assert bench.decode_bytes(lay, t, shape, stored=False)[0] == unique - B * R
    # without the cascade every request reads its whole row: unique = logical rows
    flat = _fake_layout(rows, cascade=False)
    n_rows = sum(len(r) + t + 1 for r in rows)
    assert bench.decode_bytes(flat, t, shape)[0] == n_rows * (R + 4) + qo + B * R


def test_extend_flops_count_the_unmasked_pairs():
    shape = GQA_32_8
    first = np.array([0, 13, 200, 63], np.int64)   # cached prefix P per request
    L = np.array([1, 40, 264, 64], np.int64)       # prompt length
    pairs = 0
    for P, n in zip(first, L):
        q_pos = np.arange(P, n)[:, None]           # the new tokens' positions
        k_pos = np.arange(n)[None, :]
        pairs += int((k_pos <= q_pos).sum())
    lay = SimpleNamespace(first=first, L=L)
    assert bench.extend_flops(lay, shape) == 4 * shape.head_dim_k * shape.q_heads * pairs


class _Proc:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0

    def kill(self):
        pass


def _line(sm, mx, hw="Not Active", hwt="Not Active", swt="Not Active", pc="Not Active"):
    return f"0, {sm}, {mx}, 812.40, 0x0000000000000000, {hw}, {hwt}, {swt}, {pc}"


def test_clock_sampler_median_and_reasons():
    cs = bench.ClockSampler(0)
    cs.proc = _Proc()
    cs.lines = [_line(2070, 2070), _line(1965, 2070, pc="Active"), _line(2062, 2070), "garbage line",
                _line("[N/A]", 2070), _line(2040, 2070)]
    got = cs.stop()
    assert got["samples"] == 4
    assert got["sm_mhz"] == pytest.approx((2040 + 2062) / 2)
    assert got["sm_max_mhz"] == 2070
    assert got["reasons"] == ["sw_power_cap"]
    cs.lines = [_line(1500, 2070, hw="Active"), _line(1490, 2070, hwt="Active", swt="Active")]
    got = cs.stop()
    assert got["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_sampler_without_nvidia_smi():
    cs = bench.ClockSampler(0)
    got = cs.stop()
    assert got["sm_mhz"] is None and got["reasons"] == ["nvidia-smi unavailable"]


def test_peaks_come_from_the_measured_file():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        pytest.skip("no measured peaks in this checkout")
    with open(path) as f:
        p = json.load(f)
    hbm, bf16, bf16_sus, src = bench.peaks()
    assert src == "measured"
    assert (hbm, bf16, bf16_sus) == (float(p["hbm_gbs"]), float(p["bf16_tflops"]),
                                     float(p["bf16_tflops_sustained"]))


def test_decode_summary_counts_calls_inside_timed_runs(monkeypatch):
    """Decode events may span a run of n consecutive calls (the library's
    step loop records one pair per run): the per-call time is the runs'
    total over the calls they hold, and the bytes per call the mean over
    every call inside them -- a single-call event (n = 1) and a run give the
    same figures when their calls cost the same."""
    rows = _tree_rows()
    lay = _fake_layout(rows, cascade=True)
    shape = GQA_32_8

    class Ev:
        def __init__(self, ms):
            self.ms = ms

        def elapsed_time(self, other):
            return other.ms - self.ms

    monkeypatch.setattr(bench, "peaks", lambda: (6784.8, 1904.6, 1719.1, "measured"))
    per_call_ms = 0.05
    # one run of 4 calls (t = 2..5) and one single call (t = 7)
    eng = SimpleNamespace(events={"attn_decode": [(Ev(0.0), Ev(4 * per_call_ms), ("decode", lay, 2, 4)),
                                                  (Ev(1.0), Ev(1.0 + per_call_ms), ("decode", lay, 7))]})
    summary, roof = bench.kernel_summary(eng, shape, traffic_ratio=1.5)
    d = summary["attn_decode"]
    assert d["launches"] == 5
    assert d["avg_us"] == pytest.approx(1e3 * per_call_ms)
    want = np.mean([bench.decode_bytes(lay, t, shape)[0] for t in (2, 3, 4, 5, 7)])
    assert d["bytes_per_launch"] == pytest.approx(want)
    assert roof["achieved"] == pytest.approx(want / (per_call_ms * 1e-3) / 1e9)
    assert roof["traffic"] == pytest.approx(1.5 * want)
