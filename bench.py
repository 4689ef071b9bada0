"""Benchmark: prefix-shared serving step on the few-shot workload.

Workload (one step): a batch of 256 distinct questions of 32..64 tokens behind
a cached 1792-token prefix (512-token system prompt + 5 x 256-token examples),
GQA 32 query / 8 KV heads, head_dim 128, bf16, KV pool of 2^21 slots.  One
step is the whole hot path over that batch: sched_order (longest prefix
first), rc_match_prefix + pin, rc_alloc, slot tables to the device, kv_store
+ attn_extend of the questions, rc_insert of the prompts, 128 decode steps
(attn_decode_append: the new token's K/V stored inside the cascade decode),
rc_insert of prompt + outputs and
rc_release.  Every step serves a new batch of questions (inputs already in
HBM, ~0.55 GB per step, larger than L2).

Prints one JSON line (rank 0): ``value`` with the inputs resident in HBM;
``e2e`` with every step's inputs moved from pinned host memory and its outputs
read back inside the timed region (on copy streams, overlapping the kernels);
``roofline`` of the dominant entry point against the measured peaks;
``cpu_baseline`` the oracle on the host cores (all of them, and one);
per-kernel rates and, unless ``--no-paths``, the latent (MLA) decode path, the
FP8 pool and the host tree calls.  ``--latent-only`` runs just the latent path
(smaller with ``--latent-shared/--latent-private``).  ``--impl reference``
times the CPU oracle instead, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import gc
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "prefix-shared decode attn tokens/s; HBM GB/s vs ~8 TB/s peak; prefix hit rate"
UNIT = "tokens/s"
N_QUESTIONS, MAX_NEW = 256, 128
WARM_LEN = 512 + 5 * 256


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="few_shot", choices=["few_shot", "chat", "agent", "mla"],
                    help="workload: few_shot (the default line) or one of the other configurations")
    ap.add_argument("--policy", default="lpm", choices=["lpm", "fcfs"])
    ap.add_argument("--no-cascade", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-overlap", dest="overlap", action="store_false",
                    help="serve batch by batch (no host work for batch k+1 during batch k's decode)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="budget of the oracle sample")
    ap.add_argument("--questions", type=int, default=N_QUESTIONS)
    ap.add_argument("--max-new", type=int, default=MAX_NEW)
    ap.add_argument("--pool-slots", type=int, default=0, help="KV pool size (default: the workload's 2^21)")
    ap.add_argument("--no-paths", action="store_true",
                    help="skip the per-path measurements (latent decode, host tree calls)")
    ap.add_argument("--latent-only", action="store_true",
                    help="run only the latent decode path (128 requests) and print its measurement; with "
                         "--latent-shared/--latent-private/--latent-steps a smaller case for profiling")
    ap.add_argument("--latent-shared", type=int, default=4096, help="latent path: shared prefix tokens")
    ap.add_argument("--latent-private", type=int, default=28672, help="latent path: max private tokens")
    ap.add_argument("--latent-steps", type=int, default=8, help="latent path: decode steps")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), float(p["bf16_tflops_sustained"]), "measured"
    except Exception:
        return 6800.0, 1900.0, 1700.0, "fallback"


# ----------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.th = threading.Thread(target=self._read, daemon=True)
            self.th.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def made_events(torch, n, timing=False):
    """n CUDA events, each recorded once so that the CUDA event exists (it is
    created at its first record): made before a timed region, they spare the
    region the host time of creating events."""
    evs = [torch.cuda.Event(enable_timing=timing) for _ in range(n)]
    for e in evs:
        e.record()
    torch.cuda.synchronize()
    return evs


class EventRing:
    """Ordering events handed out in turn.  An event is recorded again only
    n uses later; a stream wait queued earlier keeps the record that was
    current when it was queued, and every wait here is queued within a few
    uses of its record."""

    def __init__(self, torch, n=256):
        self.evs = made_events(torch, n)
        self.i = 0

    def __call__(self):
        e = self.evs[self.i]
        self.i = (self.i + 1) % len(self.evs)
        return e


class CopyLog:
    """CUDA events around every host<->device copy of an e2e leg, recorded on
    the copy's own stream (after its waits): how long the copies themselves
    took during the leg, to set beside the link rates measured alone."""

    def __init__(self, torch, n_copies=0):
        self.torch = torch
        self.items = []
        self.spare = made_events(torch, 2 * n_copies, timing=True)

    def _event(self):
        return self.spare.pop() if self.spare else self.torch.cuda.Event(enable_timing=True)

    def run(self, stream, kind, nbytes, fn):
        a, b = self._event(), self._event()
        a.record(stream)
        fn()
        b.record(stream)
        self.items.append((kind, nbytes, a, b))

    def summary(self, steps):
        out = {}
        for kind in ("h2d", "d2h"):
            its = [x for x in self.items if x[0] == kind]
            ms = sum(a.elapsed_time(b) for _, _, a, b in its)
            nb = sum(n for _, n, _, _ in its)
            out[kind] = {"copies_per_step": len(its) / steps, "busy_ms_per_step": ms / steps,
                         "gbs": nb / (ms * 1e-3) / 1e9 if ms > 0 else None}
        return out


# ------------------------------------------------------------ replay model
class ReplayModel:
    """The synthetic model with every step's Q/K/V rows generated ahead of time
    in the order the batch will be served (arrival order: every question
    matches the same cached prefix, so longest-prefix-first keeps arrival)."""

    def __init__(self, base, torch):
        self.base = base
        self.torch = torch
        self.ready = {}          # tuple(rids) -> dict
        self.host = None         # e2e: pinned host copies, moved to the device on use
        self.h2d_bytes = 0
        self.copylog = None      # e2e: a CopyLog timing every copy
        self._last = None        # (batch list, entry) of the batch being served

    def sequence(self, prompt, max_new):
        return self.base.sequence(prompt, max_new)

    def register(self, rid, hashes):
        self.base.register(rid, hashes)

    def hashes(self, rid):
        return self.base.hashes(rid)

    def prepare(self, reqs, first, ext_kinds=("q", "k", "v")):
        """Generate a batch's inputs in serving order.  first: the first
        computed position of every request (one int, or one per request);
        ext_kinds: the prefill rows' kinds (K only for a store without
        attention)."""
        torch = self.torch
        firsts = tuple([int(first)] * len(reqs) if np.isscalar(first) else (int(f) for f in first))
        ext_h = np.concatenate([self.base.hashes(r.rid)[f:r.prompt_len] for r, f in zip(reqs, firsts)])
        T = reqs[0].max_new
        ext = self.base.rows(ext_h, kinds=ext_kinds)
        ext = {k: ext.get(k) for k in ("q", "k", "v")}
        B = len(reqs)
        if T:
            dec_h = np.stack([self.base.hashes(r.rid)[r.prompt_len:r.prompt_len + T] for r in reqs], axis=1)
            dec = self.base.rows(dec_h.reshape(-1))
            dec = {k: (v.view(T, B, *v.shape[1:]) if v is not None else None) for k, v in dec.items()}
        else:
            dec = {}
        entry = {"ext": ext, "dec": dec, "first": firsts,
                 "dec_steps": [{k: (v[t] if v is not None else None) for k, v in dec.items()} for t in range(T)]}
        self.ready[tuple(r.rid for r in reqs)] = entry
        return entry

    # e2e: steps whose inputs move host -> device in one copy (a chunk); the
    # device holds two chunks, so chunk c+1 moves while chunk c computes
    CHUNK = 16

    def to_host(self, key):
        """e2e: keep this batch's inputs in pinned host memory only; the device
        gets them chunk by chunk on a copy stream, one chunk ahead of use."""
        torch = self.torch
        e = self.ready[key]
        pin = lambda t: t.cpu().pin_memory() if t is not None else None
        e["host"] = {"ext": {k: pin(v) for k, v in e["ext"].items()}}
        e["ext"] = {k: (torch_empty_like(torch, v)) for k, v in e["ext"].items()}
        K = self.CHUNK
        # a step's q, k and v side by side in one row of bytes (each part
        # 256-byte aligned): a chunk of steps is one contiguous copy
        dec = {k: v for k, v in e["dec"].items() if v is not None}
        T = next(iter(dec.values())).shape[0] if dec else 0
        parts, off = {}, 0
        for k, v in dec.items():
            n = v[0].numel() * v.element_size()
            parts[k] = (off, n)
            off += (n + 255) // 256 * 256
        # packed on the device, then one device -> host copy (the host buffer
        # is written by DMA, not by the CPU)
        packed = torch.zeros(T, off, dtype=torch.uint8, device=self.base.device)
        for k, v in dec.items():
            o, n = parts[k]
            packed[:, o:o + n].copy_(v.reshape(T, -1).view(torch.uint8))
        host = torch.empty(T, off, dtype=torch.uint8).pin_memory()
        host.copy_(packed)
        del packed
        e["host"]["dec"] = host
        e["dec_step_bytes"] = off
        ring = torch.empty(2 * K, off, dtype=torch.uint8, device=self.base.device)
        e["ring"] = ring
        # the step inputs as views of the ring, built once (indexing a tensor
        # costs host time on every decode step otherwise)
        e["views"] = [{k: (ring[h, parts[k][0]:parts[k][0] + parts[k][1]].view(v.dtype).view(v.shape[1:])
                           if k in dec else None) for k, v in e["dec"].items()}
                      for h in range(2 * K)]
        e["moved"] = {}          # chunk -> event on the copy stream (its copy is done)
        e["ext_moved"] = None    # event: the prefill inputs are on the device
        e["dec"] = None
        e["dec_steps"] = None

    def rearm(self):
        """e2e: every host-resident batch's inputs are to be moved again (a
        replay of the whole workload serves the same batches once more)."""
        for e in self.ready.values():
            if "host" in e:
                e["moved"] = {}
                e["ext_moved"] = None

    def start_streams(self):
        torch = self.torch
        self.h2d = torch.cuda.Stream()
        self.h2d_ext = torch.cuda.Stream()
        self.events = EventRing(torch)

    def _move_chunk(self, e, c):
        """Queue chunk c's decode inputs (steps cK..cK+K-1) into ring half c mod 2
        on the copy stream, after the compute stream is done with chunk c-2."""
        torch = self.torch
        K = self.CHUNK
        host = e["host"]["dec"]
        T = host.shape[0]
        a, b = c * K, min(T, (c + 1) * K)
        if a >= T:
            return
        free = self.events()
        free.record(torch.cuda.current_stream())
        self.h2d.wait_event(free)
        nbytes = (b - a) * e["dec_step_bytes"]

        def copy():
            with torch.cuda.stream(self.h2d):
                e["ring"][(c % 2) * K:(c % 2) * K + (b - a)].copy_(host[a:b], non_blocking=True)
        if self.copylog is not None:
            self.copylog.run(self.h2d, "h2d", nbytes, copy)
        else:
            copy()
        self.h2d_bytes += nbytes
        ev = self.events()
        ev.record(self.h2d)
        e["moved"][c] = ev

    def prefetch_extend(self, key):
        """Queue a later batch's prefill inputs on their own copy stream (they
        move while the current batch decodes), and its first chunk of decode
        inputs into its ring."""
        torch = self.torch
        e = self.ready[key]
        if "host" not in e or e["ext_moved"] is not None:
            return
        if e["host"]["dec"].shape[0] and 0 not in e["moved"]:
            self._move_chunk(e, 0)
        nbytes = sum(v.numel() * v.element_size() for v in e["ext"].values() if v is not None)

        def copy():
            with torch.cuda.stream(self.h2d_ext):
                for k, v in e["ext"].items():
                    if v is not None:
                        v.copy_(e["host"]["ext"][k], non_blocking=True)
        if self.copylog is not None:
            self.copylog.run(self.h2d_ext, "h2d", nbytes, copy)
        else:
            copy()
        self.h2d_bytes += nbytes
        ev = self.events()
        ev.record(self.h2d_ext)
        e["ext_moved"] = ev

    def _entry(self, batch):
        # the same list object is passed for every step of a batch: check it once
        if self._last is not None and self._last[0] is batch:
            return self._last[1]
        key = tuple(r.rid for r in batch)
        e = self.ready.get(key)
        if e is None or tuple(r.first for r in batch) != e["first"]:
            raise RuntimeError("batch differs from the prepared one (order or cached prefix)")
        self._last = (batch, e)
        return e

    next_key = None   # e2e: batch key -> the key served after it (its prefill inputs move early)

    def extend_inputs(self, batch):
        e = self._entry(batch)
        if "host" in e:
            key = tuple(r.rid for r in batch)
            self.prefetch_extend(key)
            self.torch.cuda.current_stream().wait_event(e["ext_moved"])
            if self.next_key is not None and self.next_key.get(key) is not None:
                self.prefetch_extend(self.next_key[key])
        return e["ext"]

    extend_kv = extend_inputs   # a store without attention reads the prepared K (and V)

    def decode_inputs(self, batch, t):
        e = self._entry(batch)
        if "host" in e:
            K = self.CHUNK
            c, i = divmod(t, K)
            if i == 0:
                if c not in e["moved"]:
                    self._move_chunk(e, c)
                self.torch.cuda.current_stream().wait_event(e["moved"][c])
                self._move_chunk(e, c + 1)   # after the compute stream's chunk c-1
            return e["views"][(c % 2) * K + i]
        return e["dec_steps"][t]


def torch_empty_like(torch, t):
    return None if t is None else torch.empty_like(t)


# -------------------------------------------------------------- algorithmic
# DRAM traffic of one attn_decode call over its algorithmic bytes, from an ncu
# capture (dram__bytes_read.sum + dram__bytes_write.sum of the cascade and the
# table-pass kernel) of this workload's decode steps 124 and 125, kernels as
# they stand: 212.39 MB and 213.51 MB of DRAM traffic for 194.72 MB and
# 195.77 MB of algorithmic bytes.  Traffic grows with the keys read, so the
# ratio scales it to the average call.
DECODE_TRAFFIC_RATIO = 1.0905
DECODE_TRAFFIC_CURRENT = True


# The same ratio for the other configurations' decode calls, from ncu
# captures (dram__bytes_read.sum + dram__bytes_write.sum of every kernel of
# three consecutive decode calls, warm-up step, kernels as they stand) over
# the bench's average algorithmic bytes per call: agent tree 520.8 MB for 3
# calls (cascade 30.5, table pass 121.3, merge 21.3 MB each) against 132.6 MB
# per call -- the split partials the merge reads are not algorithmic bytes;
# latent 5,093.7 MB for 2 calls (kernel 2,369.5, merge 177.0 MB each) against
# 2,789.7 MB per call -- the shared prefix and the rows the previous step
# left in L2 are read from L2.
CONFIG_TRAFFIC_RATIO = {"agent": 1.309, "mla": 0.913}


def row_bytes(shape):
    """K+V bytes of one token: 2 x KV heads x head_dim x 2 B; one 576-wide
    latent row (K and V share it) for the latent layout."""
    return shape.head_dim_k * 2 if shape.mla else 2 * shape.kv_heads * shape.head_dim_k * 2


def decode_bytes(lay, t, shape, stored=True):
    """Unique K/V rows touched (shared segments once) x row bytes + indices + Q + O,
    + the new token's K/V written to the pool when the call stores it (the
    latent layout stores it with kv_store inside the same timed call: read
    and written)."""
    R = row_bytes(shape)
    L = lay.L + t + 1
    tail = (L - lay.private).sum()
    seg = sum(len(s) for s, _ in lay.segments) if lay.use_cascade else 0
    B = lay.batch_size
    qo = B * shape.q_heads * (shape.head_dim_k + shape.head_dim_v) * 2
    store = (2 if shape.mla else 1) * B * R if stored else 0
    return int((seg + tail) * R + (seg + tail) * 4 + qo + store), int(L.sum() * R)


def decode_flops(lay, t, shape):
    """Scores and P.V of one decode step: 2 x Hq x (dk + dv) per key."""
    L = lay.L + t + 1
    return int(L.sum()) * 2 * shape.q_heads * (shape.head_dim_k + shape.head_dim_v)


def extend_flops(lay, shape):
    tot = 0
    for P, n in zip(lay.first, lay.L - lay.first):
        i = np.arange(n)
        tot += int((4 * shape.head_dim_k * shape.q_heads * (P + i + 1)).sum())
    return tot


def kernel_summary(eng, shape, traffic_ratio=None, traffic_note=None):
    """Per entry point: launches, time, algorithmic work and rate from the
    CUDA events recorded around its calls; the roofline object of the one
    with the largest total time (decode: HBM, and for the latent layout the
    tensor fraction beside it; extend: bf16 tensor, sustained peak since it
    runs inside a long step)."""
    hbm, bf16, bf16_sus, peak_src = peaks()
    summary = {}
    for name, evs in eng.events.items():
        if not evs:
            continue
        durs = [a.elapsed_time(b) for a, b, _ in evs]
        info = [i for _, _, i in evs]
        tot = sum(durs)
        # decode events may span a run of n steps (info[3]): averages are per call
        calls = sum(i[3] if name == "attn_decode" and len(i) > 3 else 1 for i in info)
        d = {"launches": calls, "total_ms": tot, "avg_us": 1e3 * tot / max(calls, 1)}
        sec = d["avg_us"] * 1e-6
        if name == "attn_decode":
            steps = [(i[1], t) for i in info for t in range(i[2], i[2] + (i[3] if len(i) > 3 else 1))]
            b = [decode_bytes(lay, t, shape) for lay, t in steps]
            uniq = sum(x for x, _ in b) / len(b)
            logical = sum(y for _, y in b) / len(b)
            d.update(bytes_per_launch=uniq, logical_bytes_per_launch=logical,
                     gbs=uniq / sec / 1e9, logical_gbs=logical / sec / 1e9)
            if len(steps) > len(info):
                d["timed_as"] = "runs of consecutive decode calls, one pair of events per run"
            if shape.mla:
                f = sum(decode_flops(lay, t, shape) for lay, t in steps) / len(steps)
                d.update(flops_per_launch=f, tflops=f / sec / 1e12)
        elif name == "attn_extend":
            f = sum(extend_flops(i[1], shape) for i in info) / len(info)
            d.update(flops_per_launch=f, tflops=f / sec / 1e12)
        elif name == "kv_store":
            by = sum(2 * i[1] * row_bytes(shape) for i in info) / len(info)
            d.update(bytes_per_launch=by, gbs=by / sec / 1e9)
        summary[name] = d
    dom = max(summary, key=lambda k: summary[k]["total_ms"])
    dd = summary[dom]
    if dom == "attn_extend":
        roof = {"bound": "tensor", "achieved": dd["tflops"], "peak": bf16_sus, "unit": "TFLOP/s",
                "frac": dd["tflops"] / bf16_sus, "traffic": None, "kernel": dom,
                "peak_source": f"{peak_src} bf16 dense sustained"}
    else:
        traffic = traffic_ratio * dd["bytes_per_launch"] if (dom == "attn_decode" and traffic_ratio) else None
        roof = {"bound": "hbm", "achieved": dd["gbs"], "peak": hbm, "unit": "GB/s", "frac": dd["gbs"] / hbm,
                "traffic": traffic, "kernel": dom, "peak_source": f"{peak_src} HBM copy"}
        if traffic is None and traffic_note:
            roof["traffic_note"] = traffic_note
        if dom == "attn_decode" and "tflops" in dd:   # the latent layout sits at the ridge: both fractions
            roof["tensor"] = {"achieved": dd["tflops"], "peak": bf16_sus, "unit": "TFLOP/s",
                              "frac": dd["tflops"] / bf16_sus, "peak_source": f"{peak_src} bf16 dense sustained"}
    return summary, roof


# ------------------------------------------------------------------ oracle
def oracle_baseline(trace_fn, shape, seed, vocab, budget_s, one_core=True, seed_rows=0):
    """The oracle as it stands, on a bounded sample of one step, scaled to the
    metric's unit: host tree calls of a whole step (full), attention of sampled
    extend rows and decode tokens (timed until the budget is spent)."""
    import oracle
    from radixattention_prefix_shared_tree_gb300 import workloads as wl
    from synth import hashgen as hg
    from synth.model import SynthModel
    tr = trace_fn(0)
    model = SynthModel(shape, seed, vocab, device="cpu")
    tree = oracle.OracleTree(1 << 21)
    runner = wl.Runner(tree, model, sched=oracle.OracleServer(tree))
    runner.serve([runner.request(tr.warm, 0)])
    reqs = [runner.request(tr.prompt(i), tr.max_new) for i in range(len(tr.questions))]
    t0 = time.perf_counter()
    admitted, _ = runner.serve(reqs)
    t_tree = time.perf_counter() - t0
    n_ext_total = sum(r.prompt_len - r.first for r in admitted)
    n_dec_total = len(admitted) * tr.max_new
    # attention sample: inputs of two requests generated once on the CPU (not timed)
    rng = np.random.default_rng(seed_rows)
    pre = []
    for r in admitted[:2]:
        h = model.hashes(r.rid)
        n = r.prompt_len + tr.max_new
        pre.append((r, hg.gen_values(h[:n], hg.KIND_K, shape.kv_heads, shape.head_dim_k),
                    hg.gen_values(h[:n], hg.KIND_V, shape.kv_heads, shape.head_dim_v),
                    hg.gen_values(h[:n], hg.KIND_Q, shape.q_heads, shape.head_dim_k)))
    t_att_ext = t_att_dec = 0.0
    n_ext = n_dec = 0
    while t_att_ext + t_att_dec < budget_s:
        r, kb, vb, qb = pre[int(rng.integers(0, len(pre)))]
        pos_dec = r.prompt_len + int(rng.integers(0, tr.max_new))
        pos_ext = np.arange(r.first, r.prompt_len)
        a = time.perf_counter()
        oracle.attention(qb[[pos_dec]], kb, vb, [0], [pos_dec + 1], shape.q_heads, shape.kv_heads,
                         shape.head_dim_k, shape.head_dim_v, shape.scale)
        b = time.perf_counter()
        t_att_dec += b - a
        n_dec += 1
        if n_dec % 16 == 1:
            oracle.attention(qb[pos_ext], kb, vb, np.zeros(len(pos_ext), np.int64), pos_ext + 1, shape.q_heads,
                             shape.kv_heads, shape.head_dim_k, shape.head_dim_v, shape.scale)
            t_att_ext += time.perf_counter() - b
            n_ext += len(pos_ext)
    est = t_tree + t_att_ext / n_ext * n_ext_total + t_att_dec / n_dec * n_dec_total
    value = n_dec_total / est
    cores = oracle.num_threads()
    if not one_core:
        sample = (f"oracle tree calls of one full step ({t_tree:.2f} s) + attention of {n_dec} decode tokens and "
                  f"{n_ext} prefill rows ({t_att_dec + t_att_ext:.1f} s) on {cores} threads, scaled to "
                  f"{n_dec_total} decode tokens and {n_ext_total} prefill rows per step")
        return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
                "est_s_per_step": est}
    # the same attention on one core (the tree calls are single-threaded
    # already): decode tokens for an eighth of the budget, then prefill rows
    # eight at a time for another eighth
    oracle.set_threads(1)
    s_ext = s_dec = 0.0
    m_ext = m_dec = 0
    try:
        while s_dec < budget_s / 8 or m_dec < 2:
            r, kb, vb, qb = pre[int(rng.integers(0, len(pre)))]
            pos_dec = r.prompt_len + int(rng.integers(0, tr.max_new))
            a = time.perf_counter()
            oracle.attention(qb[[pos_dec]], kb, vb, [0], [pos_dec + 1], shape.q_heads, shape.kv_heads,
                             shape.head_dim_k, shape.head_dim_v, shape.scale)
            s_dec += time.perf_counter() - a
            m_dec += 1
        while s_ext < budget_s / 8 or m_ext < 8:
            r, kb, vb, qb = pre[int(rng.integers(0, len(pre)))]
            pos_ext = r.first + rng.choice(r.prompt_len - r.first, size=min(8, r.prompt_len - r.first),
                                           replace=False)
            a = time.perf_counter()
            oracle.attention(qb[pos_ext], kb, vb, np.zeros(len(pos_ext), np.int64), pos_ext + 1, shape.q_heads,
                             shape.kv_heads, shape.head_dim_k, shape.head_dim_v, shape.scale)
            s_ext += time.perf_counter() - a
            m_ext += len(pos_ext)
    finally:
        oracle.set_threads(0)
    est1 = t_tree + s_ext / m_ext * n_ext_total + s_dec / m_dec * n_dec_total
    sample = (f"oracle tree calls of one full step ({t_tree:.2f} s) + attention of {n_dec} decode tokens and "
              f"{n_ext} prefill rows ({t_att_dec + t_att_ext:.1f} s) on {cores} threads, scaled to {n_dec_total} "
              f"decode tokens and {n_ext_total} prefill rows per step; on one core ({m_dec} decode tokens, "
              f"{m_ext} prefill rows, {s_dec + s_ext:.1f} s): {n_dec_total / est1:.1f} {UNIT}")
    return {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
            "value_one_core": n_dec_total / est1, "est_s_per_step": est}


# ------------------------------------------------------------ other configs
CONFIG_NAMES = ("few_shot", "chat", "agent", "mla")


def config_setup(name):
    """(trace, serving loop, runner options, workload description) of a
    configuration other than the default few-shot one."""
    from radixattention_prefix_shared_tree_gb300 import workloads as wl
    from synth import traces
    if name == "chat":
        tr = traces.chat()
        desc = ("multi-turn chat: 256 sessions x 8 turns, user turns U[128,512], 128 generated tokens per turn, "
                f"GQA 32q/8kv, head_dim 128, bf16, pool {tr.pool_slots} slots (0.75 of the working set, LRU "
                "eviction), decode batch <= 256; one step = the whole trace on an empty cache")
        return tr, lambda r, t: wl.run_chat(r, t, overlap=True), dict(cascade=True, prefill_attention=True), desc
    if name == "agent":
        tr = traces.agent_tree()
        desc = ("agent branching tree: 2048-token root, fan-out 4 to depth 3, 256-token branches, 64 leaves "
                f"decoding 256 tokens, GQA 64q/8kv, head_dim 128, bf16, pool {tr.pool_slots} slots; one step = "
                "the whole tree on an empty cache")
        return tr, lambda r, t: wl.run_agent(r, t, overlap=True), dict(cascade=True, prefill_attention=True), desc
    if name == "mla":
        tr = traces.mla_long()
        desc = ("latent long-context decode: 128 requests, 4096 shared + U[0,28672] private tokens, latent 576 "
                f"(512+64), 128 query heads, bf16, {tr.steps} decode steps, pool {tr.pool_slots} slots; one step = "
                "store the contexts, then every decode step, on an empty cache")
        return tr, lambda r, t: wl.run_mla(r, t, overlap=True), dict(cascade=False, prefill_attention=False), desc
    raise ValueError(name)


class MemoSequences:
    """The model's sequence() results recorded once (the host pre-run) and
    handed back in the same call order on every replay: a replay serves the
    same requests in the same order, and hashing every prompt again is the
    model's work, not the serving path's."""

    def __init__(self, base):
        self.base = base
        self.memo = []
        self.i = 0
        self.recording = True

    def sequence(self, prompt, max_new):
        if self.recording:
            r = self.base.sequence(prompt, max_new)
            self.memo.append((len(prompt), r))
            return r
        n, r = self.memo[self.i]
        if n != len(prompt):
            raise RuntimeError("a replay asked for another sequence than the pre-run")
        self.i += 1
        return r

    def replay(self):
        self.recording = False
        self.i = 0

    def __getattr__(self, name):
        return getattr(self.base, name)


def host_prerun(tr, fn, model, pool):
    """Run the workload's host calls alone (the library's tree, no device):
    the batches it serves, in order, with each request's first position."""
    import radixattention_prefix_shared_tree_gb300 as ra
    from radixattention_prefix_shared_tree_gb300 import workloads as wl
    from radixattention_prefix_shared_tree_gb300.driver import Scheduler
    sched = Scheduler(ra.RadixCache(pool))
    batches = []
    admit = sched.admit

    def rec(pending, policy, max_batch=None):
        a, w = admit(pending, policy, max_batch)
        if a:
            batches.append(list(a))
        return a, w

    sched.admit = rec
    fn(wl.Runner(sched.cache, model, sched=sched), tr)
    return batches


def row_work(batches):
    """Keys attended, summed over every computed row (prefill rows and decode
    tokens) of the served batches: what the oracle's attention costs scale
    with.  Returns (prefill rows, decode tokens, sum of keys)."""
    n_ext = n_dec = keys = 0
    for b in batches:
        for r in b:
            n = r.prompt_len - r.first
            n_ext += n
            keys += n * (r.first + r.prompt_len + 1) // 2
            n_dec += r.max_new
            keys += r.max_new * r.prompt_len + r.max_new * (r.max_new + 1) // 2
    return n_ext, n_dec, keys


def oracle_baseline_config(name, budget_s):
    """The oracle on a bounded sample of one step of a configuration: its
    tree with its own scheduling round over the whole workload (timed in
    full), and its attention timed on sampled rows of sampled requests, the
    cost per attended key scaled to every row the step computes."""
    import oracle
    from radixattention_prefix_shared_tree_gb300 import workloads as wl
    from synth import hashgen as hg
    from synth.model import SynthModel
    tr, fn, opts, _ = config_setup(name)
    sh = tr.shape
    model = SynthModel(sh, tr.seed, tr.vocab, device="cpu")
    served = []

    class Rec(oracle.OracleServer):
        def admit(self, pending, policy=oracle.LPM, max_batch=None):
            a, w = super().admit(pending, policy, max_batch)
            if a:
                served.append(list(a))
            return a, w

    tree = oracle.OracleTree(tr.pool_slots)
    t0 = time.perf_counter()
    fn(wl.Runner(tree, model, sched=Rec(tree)), tr)
    t_tree = time.perf_counter() - t0
    n_ext, n_dec, keys_total = row_work(served)
    rng = np.random.default_rng(0)
    dec_reqs = [r for b in served for r in b if r.max_new > 0]
    pick = [dec_reqs[i] for i in rng.choice(len(dec_reqs), size=min(3, len(dec_reqs)), replace=False)]
    pre = []
    for r in pick:
        h = model.hashes(r.rid)
        n = r.prompt_len + r.max_new
        kb = hg.gen_values(h[:n], hg.KIND_K, sh.kv_heads, sh.head_dim_k)
        vb = None if sh.mla else hg.gen_values(h[:n], hg.KIND_V, sh.kv_heads, sh.head_dim_v)
        pre.append((r, kb, vb, h))
    spent = keys = 0.0
    rows = 0
    while spent < budget_s or rows < 2:
        r, kb, vb, h = pre[int(rng.integers(0, len(pre)))]
        if opts["prefill_attention"] and rng.random() < 0.3 and r.prompt_len > r.first:
            pos = r.first + rng.choice(r.prompt_len - r.first, size=min(4, r.prompt_len - r.first), replace=False)
        else:
            pos = np.asarray([r.prompt_len + int(rng.integers(0, r.max_new))])
        qb = hg.gen_values(h[pos], hg.KIND_Q, sh.q_heads, sh.head_dim_k)
        a = time.perf_counter()
        oracle.attention(qb, kb, vb, np.zeros(len(pos), np.int64), pos + 1, sh.q_heads, sh.kv_heads,
                         sh.head_dim_k, sh.head_dim_v, sh.scale, latent=sh.mla)
        spent += time.perf_counter() - a
        keys += float((pos + 1).sum())
        rows += len(pos)
    if not opts["prefill_attention"]:   # the prefill only stores K/V: no attention rows
        n_ext_att, keys_total = 0, keys_total - sum(
            (r.prompt_len - r.first) * (r.first + r.prompt_len + 1) // 2 for b in served for r in b)
    else:
        n_ext_att = n_ext
    est = t_tree + spent / keys * keys_total
    cores = oracle.num_threads()
    sample = (f"oracle tree with its own scheduling round over the whole step ({t_tree:.2f} s, one thread) + "
              f"attention of {rows} sampled rows ({spent:.1f} s on {cores} threads), scaled by attended keys to "
              f"the step's {n_dec} decode tokens and {n_ext_att} prefill rows")
    return {"value": n_dec / est, "unit": UNIT, "cores": cores, "kind": "oracle", "sample": sample,
            "est_s_per_step": est}


class OutputsHome:
    """e2e: every output of a replay goes back to pinned host memory inside
    the timed region, on a copy stream: prefill outputs per batch, decode
    outputs a chunk of steps at a time from a ring the steps write into (a
    ring half is written again only after its copy has finished)."""

    def __init__(self, torch, runner, K, ext_rows, batch, shape):
        self.torch, self.runner, self.K = torch, runner, K
        self.stream = torch.cuda.Stream()
        self.host_ext = torch.empty(max(ext_rows, 1), shape.q_heads, shape.head_dim_v,
                                    dtype=torch.bfloat16).pin_memory()
        self.host_dec = torch.empty(K, batch, shape.q_heads, shape.head_dim_v, dtype=torch.bfloat16).pin_memory()
        self.done = [None, None]
        self.bytes = 0
        self.copylog = None      # a CopyLog timing every copy
        self.events = EventRing(torch)

    def _copy(self, nbytes, fn):
        if self.copylog is not None:
            self.copylog.run(self.stream, "d2h", nbytes, fn)
        else:
            fn()

    def _after_compute(self):
        ev = self.events()
        ev.record(self.torch.cuda.current_stream())
        self.stream.wait_event(ev)

    def on_extend(self, out):
        self._after_compute()

        def copy():
            with self.torch.cuda.stream(self.stream):
                self.host_ext[:out.shape[0]].copy_(out, non_blocking=True)
        self._copy(out.numel() * out.element_size(), copy)
        out.record_stream(self.stream)
        self.bytes += out.numel() * out.element_size()

    def on_decode(self, out, t, n_steps):
        K = self.K
        if (t + 1) % K and t + 1 != n_steps:
            return
        c = t // K
        outs = self.runner.decode_outs
        a, m = (c % 2) * K, t - c * K + 1
        self._after_compute()
        # a contiguous destination: a copy into a strided slice of pinned
        # memory goes through a staging tensor and does not return at once
        dst = self.host_dec.view(-1)[:outs[a:a + m].numel()].view(m, *outs.shape[1:])

        def copy():
            with self.torch.cuda.stream(self.stream):
                dst.copy_(outs[a:a + m], non_blocking=True)
        self._copy(m * out.numel() * out.element_size(), copy)
        outs.record_stream(self.stream)
        self.bytes += m * out.numel() * out.element_size()
        done = self.events()
        done.record(self.stream)
        self.done[c % 2] = done
        prev = self.done[(c + 1) % 2]
        if prev is not None:
            self.torch.cuda.current_stream().wait_event(prev)
        if t + 1 == n_steps:
            self.done = [None, None]


def run_config(args, name, rank, world, local):
    """One configuration other than the default: every step replays the
    whole workload on an empty cache, with its inputs generated beforehand
    in HBM (value) or held in pinned host memory and moved inside the timed
    region (e2e)."""
    import torch
    import torch.distributed as dist
    import radixattention_prefix_shared_tree_gb300 as ra
    from radixattention_prefix_shared_tree_gb300 import workloads as wl
    from radixattention_prefix_shared_tree_gb300.driver import DeviceEngine
    from synth.model import SynthModel

    dev = torch.device("cuda", local)
    tr, fn, opts, desc = config_setup(name)
    sh = tr.shape
    config = {"workload": desc, "policy": "lpm", "cascade": opts["cascade"], "scheduler": "overlapped",
              "l2": "inputs larger than L2 (every step reads the whole workload's inputs again, GBs)"}
    memo = MemoSequences(SynthModel(sh, tr.seed, tr.vocab, device=dev))
    batches = host_prerun(tr, fn, memo, tr.pool_slots)
    memo.replay()
    n_ext, n_dec, _ = row_work(batches)
    model = ReplayModel(memo, torch)
    kinds = ("q", "k", "v") if opts["prefill_attention"] else ("k", "v")
    keys = []
    for b in batches:
        model.prepare(b, [r.first for r in b], ext_kinds=kinds)
        keys.append(tuple(r.rid for r in b))
    eng = DeviceEngine(sh, tr.pool_slots, device=dev)

    def replay(hooks=None):
        memo.replay()
        runner = wl.Runner(ra.RadixCache(tr.pool_slots), model, eng, **opts)
        if hooks is not None:
            hooks.runner = runner
            runner.decode_out_slots = 2 * model.CHUNK
            runner.on_decode, runner.on_extend = hooks.on_decode, hooks.on_extend
        fn(runner, tr)
        return runner

    for _ in range(args.warmup):
        replay()
    torch.cuda.synchronize()
    assert ra.rc_sync(eng.err) == ra.RC_OK
    gc.collect()
    gc.freeze()
    rounds = len(batches)
    max_new = max(r.max_new for b in batches for r in b)
    eng.timing_every = 4
    eng.start_timing(args.steps * rounds * 2 * (max_new // 4 + 8) + 64)
    launches0 = eng.launches
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for _ in range(args.steps):
        runner = replay()
    ev1.record()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    eng.timing = False
    ms = slowest_rank(ev0.elapsed_time(ev1), world, dev)
    launches = eng.launches - launches0
    assert ra.rc_sync(eng.err) == ra.RC_OK
    st = runner.cache.stats()
    summary, roof = kernel_summary(eng, sh, CONFIG_TRAFFIC_RATIO.get(name),
                                   "null: no ncu DRAM capture of this configuration")
    value = whole_job_rate(args.steps * n_dec, world, ms)

    e2e = None
    if not args.no_e2e:
        for k in keys:
            model.to_host(k)
        model.next_key = {k: (keys[i + 1] if i + 1 < len(keys) else None) for i, k in enumerate(keys)}
        model.start_streams()
        ext_rows = max(int(model.ready[k]["host"]["ext"]["k"].shape[0]) for k in keys)
        home = OutputsHome(torch, None, model.CHUNK, ext_rows if opts["prefill_attention"] else 1,
                           max(len(b) for b in batches), sh)
        model.h2d_bytes = 0
        link0 = link_rates(torch)
        src_gbs = source_rate(torch, model, keys)
        model.copylog = home.copylog = CopyLog(torch, args.steps * rounds * 2 * (max_new // model.CHUNK + 2))
        wait0 = eng.host_wait_s
        gc.collect()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        h0 = time.perf_counter()
        worker_wait = 0.0
        for _ in range(args.steps):
            model.rearm()
            worker_wait += replay(home).worker_wait_s
        torch.cuda.current_stream().wait_stream(home.stream)
        e1.record()
        host_s = time.perf_counter() - h0
        torch.cuda.synchronize()
        assert ra.rc_sync(eng.err) == ra.RC_OK
        ems = slowest_rank(e0.elapsed_time(e1), world, dev)
        e2e = {"value": whole_job_rate(args.steps * n_dec, world, ems), "unit": UNIT,
               "h2d_bytes_per_step": model.h2d_bytes // args.steps, "d2h_bytes_per_step": home.bytes // args.steps,
               "ms_per_step": ems / args.steps, "host_queue_ms_per_step": 1e3 * host_s / args.steps}
        e2e["link"] = link_summary(link0, link_rates(torch), e2e["h2d_bytes_per_step"], e2e["d2h_bytes_per_step"])
        e2e["copies"] = model.copylog.summary(args.steps)
        e2e["link"]["input_buffers_gbs"] = src_gbs
        e2e["link"]["anon_huge_kb"] = anon_huge_kb()
        e2e["host_blocked_ms_per_step"] = 1e3 * (eng.host_wait_s - wait0) / args.steps
        e2e["host_worker_wait_ms_per_step"] = 1e3 * worker_wait / args.steps
        # the launching thread's own work: queueing time less its waits for the GPU and for the worker
        e2e["host_busy_ms_per_step"] = (e2e["host_queue_ms_per_step"] - e2e["host_blocked_ms_per_step"]
                                        - e2e["host_worker_wait_ms_per_step"])
        model.copylog = home.copylog = None

    cpu = None
    if rank == 0 and world == 1:
        import oracle
        oracle.build()
        cb = oracle_baseline_config(name, args.cpu_seconds)
        cpu = {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")}
    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": config, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "clocks": clk,
                "hit_rate": {"tokens": st["match_hit_tokens"] / max(st["match_tokens"], 1),
                             "requests": st["match_hits"] / max(st["match_calls"], 1)},
                "work_per_step": {"decode_tokens": n_dec, "prefill_rows": n_ext, "rounds": rounds,
                                  "evicted_tokens": st["evicted_tokens"]},
                "kernels": summary, "parallelism": "replicas" if world > 1 else "single"}
        print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- replicas
def link_rates(torch, nbytes: int = 256 << 20, reps: int = 3) -> dict:
    """Pinned host <-> device copy rates right now (GB/s, CUDA events): each
    direction alone and both at once on two streams.  The e2e leg moves its
    inputs and outputs over this link, which the host's other GPU and its
    users share: the rates, taken before and after the leg, say how much of
    the e2e time the link alone explains."""
    h_in = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(nbytes, dtype=torch.uint8).pin_memory()
    d_in = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    d_out = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    cur = torch.cuda.current_stream()
    streams = (torch.cuda.Stream(), torch.cuda.Stream())
    copies = (lambda: d_in.copy_(h_in, non_blocking=True), lambda: h_out.copy_(d_out, non_blocking=True))

    def run(which):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(cur)
        for i in which:
            streams[i].wait_stream(cur)
            with torch.cuda.stream(streams[i]):
                for _ in range(reps):
                    copies[i]()
        for i in which:
            cur.wait_stream(streams[i])
        b.record(cur)
        torch.cuda.synchronize()
        return reps * nbytes / (a.elapsed_time(b) * 1e-3) / 1e9

    run((0, 1))
    return {"h2d": run((0,)), "d2h": run((1,)), "both_each_way": run((0, 1))}


def anon_huge_kb():
    """The process's anonymous memory in transparent huge pages (kB), or None."""
    try:
        for ln in open("/proc/self/smaps_rollup"):
            if ln.startswith("AnonHugePages"):
                return int(ln.split()[1])
    except OSError:
        pass
    return None


def source_rate(torch, model, keys, nbytes: int = 32 << 20):
    """H2D rate (GB/s, CUDA events) reading the e2e leg's own pinned input
    buffers: the first nbytes of every batch's decode inputs, copied once.
    Set beside link_rates (fresh buffers) it tells a slow buffer from a slow
    link."""
    srcs = []
    for k in keys:
        h = model.ready[k]["host"]["dec"]
        if h.numel():
            srcs.append(h.reshape(-1)[:nbytes])
    if not srcs:
        return None
    d = torch.empty(max(x.numel() for x in srcs), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for x in srcs:
        d[:x.numel()].copy_(x, non_blocking=True)
    b.record()
    torch.cuda.synchronize()
    return sum(x.numel() for x in srcs) / (a.elapsed_time(b) * 1e-3) / 1e9


def link_summary(before: dict, after: dict, h2d_bytes: int, d2h_bytes: int) -> dict:
    """The link rates around an e2e leg and the time its copies alone need
    per step at the slower of the two readings: each direction alone, and
    both directions at once."""
    lo = {k: min(before[k], after[k]) for k in before}
    alone = max(h2d_bytes / lo["h2d"], d2h_bytes / lo["d2h"]) / 1e6
    both = max(h2d_bytes, d2h_bytes) / lo["both_each_way"] / 1e6
    return {"gbs_before": before, "gbs_after": after,
            "copy_ms_per_step": {"directions_alone": alone, "both_at_once": both}}


def slowest_rank(ms: float, world: int, device) -> float:
    """The job's time over N replicas: every rank times the same region
    (barriers on both sides) and the slowest one counts.  One all-reduce of
    a scalar; no data moves between replicas."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(ms)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, ms: float) -> float:
    """Units of all replicas per second of the slowest one (weak scaling)."""
    return units_per_rank * world / (ms / 1e3)


# -------------------------------------------------------------------- main
def latent_path(dev, hbm, bf16, peak_src, steps: int = 8, shared_len: int = 4096, private_max: int = 28672):
    """Latent (MLA) decode at its full configuration: 128 requests, a
    4,096-token shared prefix + U[0, 28,672] private tokens each, one
    576-wide latent head, 128 query heads.  The contexts are stored
    (kv_store, untimed), then `steps` decode steps run; attn_decode is timed
    with CUDA events per call.  Both rooflines: bytes (unique latent rows,
    the shared prefix once, and the rows this flat kernel actually reads)
    and flops (2 * Hq * (576 + 512) per key)."""
    import torch
    import radixattention_prefix_shared_tree_gb300 as ra
    from radixattention_prefix_shared_tree_gb300 import workloads as wl
    from radixattention_prefix_shared_tree_gb300.driver import DeviceEngine
    from synth import traces
    from synth.model import SynthModel

    tr = traces.mla_long(shared_len=shared_len, private_max=private_max, steps=steps)
    sh = tr.shape
    model = SynthModel(sh, tr.seed, tr.vocab, device=dev)
    eng = DeviceEngine(sh, tr.pool_slots, device=dev)
    cache = ra.RadixCache(tr.pool_slots)
    runner = wl.Runner(cache, model, eng, cascade=False, prefill_attention=False)
    eng.start_timing(16 * steps + 64)
    reqs = wl.run_mla(runner, tr)
    torch.cuda.synchronize()
    assert ra.rc_sync(eng.err) == ra.RC_OK
    evs = eng.events.get("attn_decode", [])
    durs = [a.elapsed_time(b) * 1e-3 for a, b, _ in evs]
    R = sh.head_dim_k * 2
    shared = len(tr.shared)
    ctx0 = np.asarray([r.prompt_len for r in reqs], np.int64)
    uniq, logical, flops = [], [], []
    for t in range(len(durs)):
        ctx = ctx0 + t + 1
        uniq.append((shared + (ctx - shared).sum()) * R)
        logical.append(ctx.sum() * R)
        flops.append(ctx.sum() * 2 * sh.q_heads * (sh.head_dim_k + sh.head_dim_v))
    sec = sum(durs) / len(durs)
    u, lg, f = np.mean(uniq), np.mean(logical), np.mean(flops)
    return {"config": "128 requests, %d shared + U[0,%d] private tokens, latent 576 (512+64), "
                      "128 query heads, bf16; %d decode steps" % (shared_len, private_max, len(durs)),
            "us_per_step": sec * 1e6, "tokens_per_s": len(reqs) / sec,
            "unique_bytes": float(u), "logical_bytes": float(lg), "flops": float(f),
            "hbm": {"achieved_unique_gbs": u / sec / 1e9, "achieved_read_gbs": lg / sec / 1e9, "peak": hbm,
                    "frac_unique": u / sec / 1e9 / hbm, "frac_read": lg / sec / 1e9 / hbm},
            "tensor": {"achieved_tflops": f / sec / 1e12, "peak": bf16, "frac": f / sec / 1e12 / bf16},
            "peak_source": f"{peak_src} HBM copy and bf16 dense burst"}


def fp8_path(dev, hbm, peak_src, trace_fn, args, steps: int = 3, warmup: int = 2):
    """The benchmark's step (same workload, same launch configuration) over an
    E4M3 pool: prefill quantises the new tokens (kv_store) and reads codes
    (tcgen05 kernel, f16 products), every decode step stores the new token's
    codes and scales (kv_store) and attends over codes (cascade + table pass).
    Timed with CUDA events around the steps; attn_decode per call on every 4th
    step (the event pair also covers that step's kv_store).  Bytes per call:
    unique rows x (codes + scale) for K and V, indices, Q, O, and the new
    token (bf16 read, codes and scales written)."""
    import torch
    import radixattention_prefix_shared_tree_gb300 as ra
    from radixattention_prefix_shared_tree_gb300 import workloads as wl
    from radixattention_prefix_shared_tree_gb300.driver import DeviceEngine
    from synth.model import SynthModel

    tr0 = trace_fn(0)
    sh = tr0.shape
    base = SynthModel(sh, tr0.seed, tr0.vocab, device=dev)
    model = ReplayModel(base, torch)
    pool = args.pool_slots or tr0.pool_slots
    eng = DeviceEngine(sh, pool, device=dev, kv_fp8=True)
    runner = wl.Runner(ra.RadixCache(pool), model, eng, cascade=True)
    runner.model = base
    runner.serve([runner.request(tr0.warm, 0)])
    runner.model = model
    batches = []
    for s in range(warmup + steps):
        tr = trace_fn(1000 + s)
        reqs = [runner.request(tr.prompt(i), tr.max_new) for i in range(len(tr.questions))]
        model.prepare(reqs, WARM_LEN)
        batches.append(reqs)
    for s in range(warmup):
        runner.serve(batches[s])
    torch.cuda.synchronize()
    eng.timing_every = 4
    eng.start_timing(4 * steps * (args.max_new + 8) + 64)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record()
    for s in range(warmup, warmup + steps):
        runner.serve(batches[s])
    ev1.record()
    torch.cuda.synchronize()
    assert ra.rc_sync(eng.err) == ra.RC_OK
    ms = ev0.elapsed_time(ev1) / steps
    R8 = 2 * sh.kv_heads * (sh.head_dim_k + 4)
    evs = eng.events.get("attn_decode", [])
    durs = [a.elapsed_time(b) * 1e-3 for a, b, _ in evs]
    by = []
    calls = 0
    for _, _, info in evs:
        n = info[3] if len(info) > 3 else 1    # an event pair may span a run of n steps
        calls += n
        for t in range(info[2], info[2] + n):
            lay = info[1]
            L = lay.L + t + 1
            tail = (L - lay.private).sum()
            seg = sum(len(x) for x, _ in lay.segments) if lay.use_cascade else 0
            B = lay.batch_size
            qo = B * sh.q_heads * (sh.head_dim_k + sh.head_dim_v) * 2
            store = B * (2 * sh.kv_heads * sh.head_dim_k * 2 + R8)
            by.append((seg + tail) * R8 + (seg + tail) * 4 + qo + store)
    sec = sum(durs) / max(calls, 1)
    u = float(np.mean(by)) if by else 0.0
    ext = eng.events.get("attn_extend", [])
    ext_us = 1e3 * sum(a.elapsed_time(b) for a, b, _ in ext) / max(len(ext), 1)
    return {"config": "the benchmark's workload and launch configuration over an E4M3 pool "
                      "(one fp32 scale per (slot, KV head) row); %d timed steps" % steps,
            "tokens_per_s": args.questions * args.max_new / (ms * 1e-3), "ms_per_step": ms,
            "attn_decode_us": sec * 1e6, "attn_extend_us": ext_us, "bytes_per_call": u,
            "hbm": {"achieved_gbs": u / sec / 1e9, "peak": hbm, "frac": u / sec / 1e9 / hbm},
            "peak_source": f"{peak_src} HBM copy"}


def main():
    args = parse()
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from synth import traces
    trace_fn = lambda salt: traces.few_shot(n_questions=args.questions, max_new=args.max_new, batch_salt=salt)
    tr0 = trace_fn(0)
    shape = tr0.shape
    config = {"workload": f"few-shot sharing: {WARM_LEN}-token shared prefix (512 system + 5x256 examples), "
                          f"{args.questions} questions U[32,64], {args.max_new} decode steps, "
                          "GQA 32q/8kv, head_dim 128, bf16, pool 2^21 slots",
              "policy": args.policy, "cascade": not args.no_cascade,
              "scheduler": "overlapped" if args.overlap else "serial",
              "l2": "inputs larger than L2 (a new batch per step, ~0.55 GB of Q/K/V each)"}

    if args.impl == "reference" and args.config != "few_shot":
        if rank != 0:
            return
        import oracle
        oracle.build()
        cb = oracle_baseline_config(args.config, max(args.cpu_seconds, 5.0))
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": 0,
                "steps": 1, "extrapolated": True, "warmup": 0, "ms_per_step": cb["est_s_per_step"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": {"workload": config_setup(args.config)[3]},
                "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample")},
                "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return
    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        # every step (warm-up included) is one bounded sample of a step: the
        # oracle tree's calls of a whole step and attention of sampled rows,
        # scaled to the step; the timed steps' estimates are averaged
        per = max(args.cpu_seconds / max(args.steps, 1), 0.4)
        ests, cb = [], None
        for s_ in range(args.warmup + args.steps):
            cb = oracle_baseline(trace_fn, shape, tr0.seed, tr0.vocab, per, one_core=False, seed_rows=s_)
            if s_ >= args.warmup:
                ests.append(cb["est_s_per_step"])
        est = float(np.mean(ests))
        tokens = args.questions * args.max_new
        sample = (f"{args.steps} timed steps (+{args.warmup} warm-up), each a bounded sample of one step "
                  f"(~{per:.1f} s of attention); the last: {cb['sample']}")
        line = {"impl": "reference", "metric": METRIC, "value": tokens / est, "unit": UNIT, "n_gpus": 0,
                "steps": args.steps, "extrapolated": True, "warmup": args.warmup, "ms_per_step": est * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {"value": tokens / est, "unit": UNIT, "cores": cb["cores"], "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": tokens / est, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
        print(json.dumps(line), flush=True)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)

    import __graft_entry__
    __graft_entry__.build()
    if args.config != "few_shot":
        run_config(args, args.config, rank, world, local)
        if world > 1:
            dist.destroy_process_group()
        return
    if args.latent_only:
        hbm, bf16, _, peak_src = peaks()
        print(json.dumps(latent_path(dev, hbm, bf16, peak_src, steps=args.latent_steps,
                                     shared_len=args.latent_shared, private_max=args.latent_private)), flush=True)
        return
    import radixattention_prefix_shared_tree_gb300 as ra
    from radixattention_prefix_shared_tree_gb300 import workloads as wl
    from radixattention_prefix_shared_tree_gb300.driver import DeviceEngine
    from synth.model import SynthModel

    policy = ra.RC_LPM if args.policy == "lpm" else ra.RC_FCFS
    base = SynthModel(shape, tr0.seed, tr0.vocab, device=dev)
    model = ReplayModel(base, torch)
    pool_slots = args.pool_slots or tr0.pool_slots
    if args.pool_slots:
        config["pool_slots"] = pool_slots
    eng = DeviceEngine(shape, pool_slots, device=dev)
    cache = ra.RadixCache(pool_slots)
    runner = wl.Runner(cache, model, eng, policy=policy, cascade=not args.no_cascade)
    # warm prefix cached (setup, untimed)
    runner.model = base
    runner.serve([runner.request(tr0.warm, 0)])
    runner.model = model

    n_main = args.warmup + args.steps
    n_e2e = 0 if args.no_e2e else args.steps
    batches = []
    for s in range(n_main + n_e2e):
        tr = trace_fn(s + 1)
        reqs = [runner.request(tr.prompt(i), tr.max_new) for i in range(len(tr.questions))]
        model.prepare(reqs, WARM_LEN)
        batches.append(reqs)
    torch.cuda.synchronize()

    def step(reqs):
        admitted, waiting = runner.serve(reqs)
        if waiting or len(admitted) != len(reqs):
            raise RuntimeError("batch did not fit")
        return admitted

    def serve_steps(lo, hi):
        """Steps lo..hi-1, one batch each: with the overlapped scheduler (the
        default) a batch's admission runs on the worker thread while the
        previous batch's decode steps are launched."""
        if not args.overlap:
            for s_ in range(lo, hi):
                step(batches[s_])
                batches[s_] = None
            return
        cur = [lo]

        def after(admitted, waiting):
            if waiting or len(admitted) != len(batches[cur[0]]):
                raise RuntimeError("batch did not fit")
            batches[cur[0]] = None
            cur[0] += 1
            return batches[cur[0]] if cur[0] < hi else None

        runner.serve_rounds(batches[lo], after, None, overlap=True)

    # a served batch is dropped at once, as a serving loop would: its slot
    # rows' memory goes back to the allocator (fresh pages cost the next
    # admission round page faults)
    serve_steps(0, args.warmup)
    torch.cuda.synchronize()
    assert ra.rc_sync(eng.err) == ra.RC_OK

    # host time of the tree calls (one admission round, prompt commit and
    # finish per step, each over the whole batch), per request
    host_t = {"admit": 0.0, "commit_prompts": 0.0, "finish": 0.0}

    def timed(name, fn):
        def g(*a, **k):
            t = time.perf_counter()
            try:
                return fn(*a, **k)
            finally:
                host_t[name] += time.perf_counter() - t
        return g

    # The objects built so far (prepared inputs, requests, traces) live for
    # the whole run: move them out of the cyclic collector's reach, as a
    # serving process does after warm-up, so a full collection does not land
    # inside a timed step.
    gc.collect()
    gc.freeze()

    # ---------------------------------------------------------- timed region
    # per-kernel durations: CUDA events around every call of the prefill and
    # around every 4th decode step (recording them costs host time per call)
    eng.timing_every = 4
    eng.start_timing(4 * (args.steps * (args.max_new * 3 + 8)) + 64)
    launches0 = eng.launches
    st0 = cache.stats()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sched_calls = {n: getattr(runner.sched, n) for n in host_t}
    for n, fn in sched_calls.items():
        setattr(runner.sched, n, timed(n, fn))
    w0 = time.perf_counter()
    ev0.record()
    serve_steps(args.warmup, n_main)
    ev1.record()
    torch.cuda.synchronize()
    wall = time.perf_counter() - w0
    if world > 1:
        dist.barrier()
    clk = clocks.stop()
    eng.timing = False
    ms = slowest_rank(ev0.elapsed_time(ev1), world, dev)
    launches = eng.launches - launches0
    st1 = cache.stats()
    assert ra.rc_sync(eng.err) == ra.RC_OK

    tokens = args.steps * args.questions * args.max_new
    value = whole_job_rate(tokens, world, ms)

    # per-call durations (events on the launching stream)
    hbm, bf16, bf16_sus, peak_src = peaks()
    note = (f"null: the last ncu capture (steps 124-125) measured {DECODE_TRAFFIC_RATIO} x the algorithmic bytes, "
            "before the cascade kernel moved its grid-dependency wait behind its reads (no memory access "
            "changed); not yet captured again")
    summary, roof = kernel_summary(eng, shape, DECODE_TRAFFIC_RATIO if DECODE_TRAFFIC_CURRENT else None,
                                   None if DECODE_TRAFFIC_CURRENT else note)

    hit_tok = (st1["match_hit_tokens"] - st0["match_hit_tokens"]) / max(st1["match_tokens"] - st0["match_tokens"], 1)
    hit_req = (st1["match_hits"] - st0["match_hits"]) / max(st1["match_calls"] - st0["match_calls"], 1)

    # ------------------------------------------------------------------ e2e
    e2e = None
    if n_e2e:
        keys = []
        for s in range(n_main, n_main + n_e2e):
            key = tuple(r.rid for r in batches[s])
            model.to_host(key)
            keys.append(key)
        torch.cuda.synchronize()
        # Inputs move host -> device on copy streams one chunk (16 steps) ahead,
        # the next batch's prefill inputs during this batch's decode; outputs
        # move device -> host on a third stream, a chunk at a time from a ring
        # the decode steps write into (the ring half is reused only after its
        # copy has finished).  Every byte of every step crosses inside the
        # timed region; the copies overlap the kernels instead of queueing
        # behind them.
        model.start_streams()
        d2h_stream = torch.cuda.Stream()
        K = model.CHUNK
        runner.decode_out_slots = 2 * K
        d2h = [0]
        st = {"batch": 0, "done": [None, None]}
        # pinned output buffers, allocated once before the timed region (a
        # page-locked allocation costs milliseconds): the largest prefill
        # output of these batches and one chunk of decode outputs
        sh = shape
        ext_rows = max(model.ready[k]["host"]["ext"]["q"].shape[0] for k in keys)
        host_ext = torch.empty(ext_rows, sh.q_heads, sh.head_dim_v, dtype=torch.bfloat16).pin_memory()
        host_dec = torch.empty(K, args.questions, sh.q_heads, sh.head_dim_v, dtype=torch.bfloat16).pin_memory()

        events = EventRing(torch)

        def after_compute():
            ev = events()
            ev.record(torch.cuda.current_stream())
            d2h_stream.wait_event(ev)

        # copies per step: a chunk of decode inputs and of outputs per K steps, the prefill's both ways
        copylog = CopyLog(torch, n_e2e * 2 * (args.max_new // model.CHUNK + 2))

        def copy_extend(out):
            after_compute()

            def copy():
                with torch.cuda.stream(d2h_stream):
                    host_ext[:out.shape[0]].copy_(out, non_blocking=True)
            copylog.run(d2h_stream, "d2h", out.numel() * out.element_size(), copy)
            out.record_stream(d2h_stream)
            d2h[0] += out.numel() * out.element_size()
            if st["batch"] + 1 < len(keys):
                model.prefetch_extend(keys[st["batch"] + 1])

        def copy_decode(out, t, n_steps):
            if (t + 1) % K and t + 1 != n_steps:
                return
            c = t // K
            outs = runner.decode_outs
            a, m = (c % 2) * K, t - c * K + 1
            after_compute()

            def copy():
                with torch.cuda.stream(d2h_stream):
                    host_dec[:m].copy_(outs[a:a + m], non_blocking=True)
            copylog.run(d2h_stream, "d2h", m * out.numel() * out.element_size(), copy)
            outs.record_stream(d2h_stream)
            d2h[0] += m * out.numel() * out.element_size()
            done = events()
            done.record(d2h_stream)
            st["done"][c % 2] = done
            # chunk c+1 writes the other ring half: chunk c-1's copy must be done
            prev = st["done"][(c + 1) % 2]
            if prev is not None:
                torch.cuda.current_stream().wait_event(prev)
            if t + 1 == n_steps:
                st["batch"] += 1
                st["done"] = [None, None]

        runner.on_decode = copy_decode
        runner.on_extend = copy_extend
        model.h2d_bytes = 0
        link0 = link_rates(torch)
        src_gbs = source_rate(torch, model, keys)
        model.copylog = copylog
        wait0, ww0 = eng.host_wait_s, runner.worker_wait_s
        gc.collect()
        gc.freeze()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        h0 = time.perf_counter()
        serve_steps(n_main, n_main + n_e2e)
        torch.cuda.current_stream().wait_stream(d2h_stream)
        e1.record()
        host_s = time.perf_counter() - h0   # time the host took to queue the work
        torch.cuda.synchronize()
        runner.on_decode = runner.on_extend = None
        runner.decode_out_slots = 1
        ems = slowest_rank(e0.elapsed_time(e1), world, dev)
        e2e = {"value": whole_job_rate(n_e2e * args.questions * args.max_new, world, ems), "unit": UNIT,
               "h2d_bytes_per_step": model.h2d_bytes // n_e2e, "d2h_bytes_per_step": d2h[0] // n_e2e,
               "ms_per_step": ems / n_e2e, "host_queue_ms_per_step": 1e3 * host_s / n_e2e}
        e2e["link"] = link_summary(link0, link_rates(torch), e2e["h2d_bytes_per_step"], e2e["d2h_bytes_per_step"])
        e2e["copies"] = copylog.summary(n_e2e)
        e2e["link"]["input_buffers_gbs"] = src_gbs
        e2e["link"]["anon_huge_kb"] = anon_huge_kb()
        e2e["host_blocked_ms_per_step"] = 1e3 * (eng.host_wait_s - wait0) / n_e2e
        e2e["host_worker_wait_ms_per_step"] = 1e3 * (runner.worker_wait_s - ww0) / n_e2e
        # the launching thread's own work: queueing time less its waits for the GPU and for the worker
        e2e["host_busy_ms_per_step"] = (e2e["host_queue_ms_per_step"] - e2e["host_blocked_ms_per_step"]
                                        - e2e["host_worker_wait_ms_per_step"])
        model.copylog = None

    cpu = None
    if rank == 0 and world == 1:
        import oracle
        oracle.build()
        cpu = oracle_baseline(trace_fn, shape, tr0.seed, tr0.vocab, args.cpu_seconds)
        cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample", "value_one_core")}

    for n, fn in sched_calls.items():
        setattr(runner.sched, n, fn)
    paths = None
    if rank == 0 and not args.no_paths:
        n_req = args.steps * args.questions
        paths = {"host_tree_us_per_request": {n: 1e6 * v / n_req for n, v in host_t.items()},
                 "latent_decode": latent_path(dev, hbm, bf16, peak_src),
                 "fp8_kv": fp8_path(dev, hbm, peak_src, trace_fn, args)}

    if rank == 0:
        line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": config, "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
                "clocks": clk, "hit_rate": {"tokens": hit_tok, "requests": hit_req},
                "kernels": summary, "paths": paths, "wall_s_timed": wall,
                "parallelism": "replicas" if world > 1 else "single"}
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
