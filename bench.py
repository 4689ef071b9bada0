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
    ap.add_argument("--policy", default="lpm", choices=["lpm", "fcfs"])
    ap.add_argument("--no-cascade", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
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
        self._last = None        # (batch list, entry) of the batch being served

    def sequence(self, prompt, max_new):
        return self.base.sequence(prompt, max_new)

    def register(self, rid, hashes):
        self.base.register(rid, hashes)

    def hashes(self, rid):
        return self.base.hashes(rid)

    def prepare(self, reqs, first: int):
        torch = self.torch
        ext_h = np.concatenate([self.base.hashes(r.rid)[first:r.prompt_len] for r in reqs])
        T = reqs[0].max_new
        dec_h = np.stack([self.base.hashes(r.rid)[r.prompt_len:r.prompt_len + T] for r in reqs], axis=1)
        ext = self.base.rows(ext_h)
        dec = self.base.rows(dec_h.reshape(-1))
        B = len(reqs)
        dec = {k: (v.view(T, B, *v.shape[1:]) if v is not None else None) for k, v in dec.items()}
        entry = {"ext": ext, "dec": dec, "first": first,
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
        e["host"] = {"ext": {k: pin(v) for k, v in e["ext"].items()},
                     "dec": {k: pin(v) for k, v in e["dec"].items()}}
        e["ext"] = {k: (torch_empty_like(torch, v)) for k, v in e["ext"].items()}
        K = self.CHUNK
        e["ring"] = {k: (torch.empty((2 * K,) + tuple(v.shape[1:]), dtype=v.dtype, device=v.device)
                         if v is not None else None) for k, v in e["dec"].items()}
        # the step inputs as views of the ring, built once (indexing a tensor
        # costs host time on every decode step otherwise)
        e["views"] = [{k: (ring[h] if ring is not None else None) for k, ring in e["ring"].items()}
                      for h in range(2 * K)]
        e["moved"] = {}          # chunk -> event on the copy stream (its copy is done)
        e["ext_moved"] = None    # event: the prefill inputs are on the device
        e["dec"] = None
        e["dec_steps"] = None

    def start_streams(self):
        torch = self.torch
        self.h2d = torch.cuda.Stream()
        self.h2d_ext = torch.cuda.Stream()

    def _move_chunk(self, e, c):
        """Queue chunk c's decode inputs (steps cK..cK+K-1) into ring half c mod 2
        on the copy stream, after the compute stream is done with chunk c-2."""
        torch = self.torch
        K = self.CHUNK
        T = next(v for v in e["host"]["dec"].values() if v is not None).shape[0]
        a, b = c * K, min(T, (c + 1) * K)
        if a >= T:
            return
        free = torch.cuda.Event()
        free.record(torch.cuda.current_stream())
        self.h2d.wait_event(free)
        with torch.cuda.stream(self.h2d):
            for k, ring in e["ring"].items():
                if ring is not None:
                    src = e["host"]["dec"][k][a:b]
                    ring[(c % 2) * K:(c % 2) * K + (b - a)].copy_(src, non_blocking=True)
                    self.h2d_bytes += src.numel() * src.element_size()
        ev = torch.cuda.Event()
        ev.record(self.h2d)
        e["moved"][c] = ev

    def prefetch_extend(self, key):
        """Queue a later batch's prefill inputs on their own copy stream (they
        move while the current batch decodes)."""
        torch = self.torch
        e = self.ready[key]
        if "host" not in e or e["ext_moved"] is not None:
            return
        with torch.cuda.stream(self.h2d_ext):
            for k, v in e["ext"].items():
                if v is not None:
                    v.copy_(e["host"]["ext"][k], non_blocking=True)
                    self.h2d_bytes += v.numel() * v.element_size()
        ev = torch.cuda.Event()
        ev.record(self.h2d_ext)
        e["ext_moved"] = ev

    def _entry(self, batch):
        # the same list object is passed for every step of a batch: check it once
        if self._last is not None and self._last[0] is batch:
            return self._last[1]
        key = tuple(r.rid for r in batch)
        e = self.ready.get(key)
        if e is None or any(r.first != e["first"] for r in batch):
            raise RuntimeError("batch differs from the prepared one (order or cached prefix)")
        self._last = (batch, e)
        return e

    def extend_inputs(self, batch):
        e = self._entry(batch)
        if "host" in e:
            key = tuple(r.rid for r in batch)
            self.prefetch_extend(key)
            self.torch.cuda.current_stream().wait_event(e["ext_moved"])
        return e["ext"]

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
# table-pass kernel) of this workload's decode steps 125 and 126: 211.78 MB and
# 212.95 MB of DRAM traffic for 195.77 MB and 196.82 MB of algorithmic bytes.
# Traffic grows with the keys read, so the ratio scales it to the average call.
# That capture predates the cascade kernel's CTA-wide barrier at entry (no
# memory access added or removed); until the counters are taken again on the
# kernel as it stands, the line reports traffic as null and this ratio in a
# note.
DECODE_TRAFFIC_RATIO = 1.0818
DECODE_TRAFFIC_CURRENT = False


def decode_bytes(lay, t, shape, stored=True):
    """Unique K/V rows touched (shared segments once) x row bytes + indices + Q + O,
    + the new token's K/V written to the pool when the call stores it."""
    R = 2 * shape.kv_heads * shape.head_dim_k * 2
    L = lay.L + t + 1
    tail = (L - lay.private).sum()
    seg = sum(len(s) for s, _ in lay.segments) if lay.use_cascade else 0
    B = lay.batch_size
    qo = B * shape.q_heads * (shape.head_dim_k + shape.head_dim_v) * 2
    store = B * R if stored else 0
    return int((seg + tail) * R + (seg + tail) * 4 + qo + store), int(L.sum() * R)


def extend_flops(lay, shape):
    tot = 0
    for P, n in zip(lay.first, lay.L - lay.first):
        i = np.arange(n)
        tot += int((4 * shape.head_dim_k * shape.q_heads * (P + i + 1)).sum())
    return tot


# ------------------------------------------------------------------ oracle
def oracle_baseline(trace_fn, shape, seed, vocab, budget_s):
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
    runner = wl.Runner(tree, model)
    runner.serve([runner.request(tr.warm, 0)])
    reqs = [runner.request(tr.prompt(i), tr.max_new) for i in range(len(tr.questions))]
    t0 = time.perf_counter()
    admitted, _ = runner.serve(reqs)
    t_tree = time.perf_counter() - t0
    n_ext_total = sum(r.prompt_len - r.first for r in admitted)
    n_dec_total = len(admitted) * tr.max_new
    # attention sample: inputs of two requests generated once on the CPU (not timed)
    rng = np.random.default_rng(0)
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


# ---------------------------------------------------------------- replicas
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
    for _, _, info in evs:
        lay, t = info[1], info[2]
        L = lay.L + t + 1
        tail = (L - lay.private).sum()
        seg = sum(len(x) for x, _ in lay.segments) if lay.use_cascade else 0
        B = lay.batch_size
        qo = B * sh.q_heads * (sh.head_dim_k + sh.head_dim_v) * 2
        store = B * (2 * sh.kv_heads * sh.head_dim_k * 2 + R8)
        by.append((seg + tail) * R8 + (seg + tail) * 4 + qo + store)
    sec = sum(durs) / max(len(durs), 1)
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
              "l2": "inputs larger than L2 (a new batch per step, ~0.55 GB of Q/K/V each)"}

    if args.impl == "reference":
        if rank != 0:
            return
        import oracle
        oracle.build()
        cb = oracle_baseline(trace_fn, shape, tr0.seed, tr0.vocab, max(args.cpu_seconds, 5.0))
        steps_t = []
        for _ in range(args.warmup + args.steps):
            steps_t.append(cb["est_s_per_step"])
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": UNIT, "n_gpus": 0,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": cb["est_s_per_step"] * 1e3,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                "data": "synthetic", "config": config,
                "cpu_baseline": {k: cb[k] for k in ("value", "unit", "cores", "kind", "sample", "value_one_core")},
                "e2e": {"value": cb["value"], "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
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

    # a served batch is dropped at once, as a serving loop would: its slot
    # rows' memory goes back to the allocator (fresh pages cost the next
    # admission round page faults)
    for s in range(args.warmup):
        step(batches[s])
        batches[s] = None
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
    for s in range(args.warmup, n_main):
        step(batches[s])
        batches[s] = None
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
    calls = {}
    for name, evs in eng.events.items():
        durs = [a.elapsed_time(b) for a, b, _ in evs]
        info = [i for _, _, i in evs]
        calls[name] = (durs, info)
    summary = {}
    for name, (durs, info) in calls.items():
        tot = sum(durs)
        d = {"launches": len(durs), "total_ms": tot, "avg_us": 1e3 * tot / max(len(durs), 1)}
        if name == "attn_decode":
            b = [decode_bytes(i[1], i[2], shape) for i in info]
            uniq = sum(x for x, _ in b) / len(b)
            logical = sum(y for _, y in b) / len(b)
            d.update(bytes_per_launch=uniq, logical_bytes_per_launch=logical,
                     gbs=uniq / (d["avg_us"] * 1e-6) / 1e9, logical_gbs=logical / (d["avg_us"] * 1e-6) / 1e9)
        elif name == "attn_extend":
            f = sum(extend_flops(i[1], shape) for i in info) / len(info)
            d.update(flops_per_launch=f, tflops=f / (d["avg_us"] * 1e-6) / 1e12)
        elif name == "kv_store":
            R = 2 * shape.kv_heads * shape.head_dim_k * 2
            by = sum(2 * i[1] * R for i in info) / len(info)
            d.update(bytes_per_launch=by, gbs=by / (d["avg_us"] * 1e-6) / 1e9)
        summary[name] = d
    dom = max(summary, key=lambda k: summary[k]["total_ms"])
    dd = summary[dom]
    if dom == "attn_extend":
        roof = {"bound": "tensor", "achieved": dd["tflops"], "peak": bf16_sus, "unit": "TFLOP/s",
                "frac": dd["tflops"] / bf16_sus, "traffic": None, "kernel": dom,
                "peak_source": f"{peak_src} bf16 dense sustained"}
    else:
        traffic = (DECODE_TRAFFIC_RATIO * dd["bytes_per_launch"]
                   if dom == "attn_decode" and DECODE_TRAFFIC_CURRENT else None)
        roof = {"bound": "hbm", "achieved": dd["gbs"], "peak": hbm, "unit": "GB/s", "frac": dd["gbs"] / hbm,
                "traffic": traffic, "kernel": dom, "peak_source": f"{peak_src} HBM copy"}
        if dom == "attn_decode" and not DECODE_TRAFFIC_CURRENT:
            roof["traffic_note"] = (f"null: the last ncu capture (steps 125-126) measured {DECODE_TRAFFIC_RATIO} x "
                                    "the algorithmic bytes, before the cascade kernel gained a CTA-wide barrier at "
                                    "entry (no memory access changed); not yet captured again")

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

        def after_compute():
            ev = torch.cuda.Event()
            ev.record(torch.cuda.current_stream())
            d2h_stream.wait_event(ev)

        def copy_extend(out):
            after_compute()
            with torch.cuda.stream(d2h_stream):
                host_ext[:out.shape[0]].copy_(out, non_blocking=True)
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
            with torch.cuda.stream(d2h_stream):
                host_dec[:m].copy_(outs[a:a + m], non_blocking=True)
            outs.record_stream(d2h_stream)
            d2h[0] += m * out.numel() * out.element_size()
            done = torch.cuda.Event()
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
        gc.collect()
        gc.freeze()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        h0 = time.perf_counter()
        for s in range(n_main, n_main + n_e2e):
            step(batches[s])
            batches[s] = None
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
