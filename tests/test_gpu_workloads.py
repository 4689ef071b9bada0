"""Workloads end to end on the GPU through the C-ABI, against the oracle.

The oracle side never sees the pool or the tree: for a request it regenerates
K/V of every position of the request's own token sequence from the prefix
hash (the cache-disabled definition) and computes attention from them.  So a
wrong match, a wrong slot, a lost duplicate or a bad eviction shows up as a
numeric mismatch.  Hit counts and slot indices are compared bit for bit with
the oracle tree running the same trace.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import radixattention_prefix_shared_tree_gb300 as ra
from radixattention_prefix_shared_tree_gb300 import workloads as wl
from radixattention_prefix_shared_tree_gb300.driver import DeviceEngine
from synth import hashgen as hg
from synth import traces
from synth.model import SynthModel
from tests import tolerance as tol

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = tol.MAX_ABS, tol.MEAN_ABS, tol.LSE_ABS


def oracle_positions(shape, hashes, positions, fp8=False):
    """Oracle attention for query positions of one request (keys 0..pos):
    (out, lse, A), A = the same attention over |V| (the bound's weight).
    fp8: K/V as an FP8 pool holds them (the oracle's own quantisation)."""
    n = int(max(positions)) + 1
    kb = hg.gen_values(hashes[:n], hg.KIND_K, shape.kv_heads, shape.head_dim_k)
    vb = None if shape.mla else hg.gen_values(hashes[:n], hg.KIND_V, shape.kv_heads, shape.head_dim_v)
    qb = hg.gen_values(hashes[np.asarray(positions)], hg.KIND_Q, shape.q_heads, shape.head_dim_k)
    zeros, ctx = np.zeros(len(positions), np.int64), np.asarray(positions, np.int64) + 1
    if fp8:
        from oracle import fp8_oracle as f8
        kd = f8.dequantize(*f8.quantize_rows(kb.reshape(n, shape.kv_heads, -1)))
        vd = f8.dequantize(*f8.quantize_rows(vb.reshape(n, shape.kv_heads, -1)))
        qr = qb.reshape(len(positions), shape.q_heads, -1)
        out, lse = f8.attention(qr, kd, vd, zeros, ctx, shape.q_heads, shape.kv_heads, shape.scale)
        a_abs, _ = f8.attention(qr, kd, np.abs(vd), zeros, ctx, shape.q_heads, shape.kv_heads, shape.scale)
        return out, lse, a_abs
    out, lse = oracle.attention(qb, kb, vb, zeros, ctx, shape.q_heads, shape.kv_heads, shape.head_dim_k,
                                shape.head_dim_v, shape.scale, latent=shape.mla)
    if shape.mla:   # V = the first head_dim_v columns of the latent row
        k3 = kb.reshape(n, 1, shape.head_dim_k)
        va = tol.abs_bits(k3[:, :, :shape.head_dim_v])
        a_abs, _ = oracle.attention(qb, k3, va, zeros, ctx, shape.q_heads, 1, shape.head_dim_k, shape.head_dim_v,
                                    shape.scale)
    else:
        a_abs, _ = oracle.attention(qb, kb, tol.abs_bits(vb), zeros, ctx, shape.q_heads, shape.kv_heads,
                                    shape.head_dim_k, shape.head_dim_v, shape.scale)
    return out, lse, a_abs


def compare(out_bits, lse, refs, stats, fp8=False):
    """Elementwise bound of tests/tolerance.py; the mean bound is checked by
    the caller over all compared elements (stats)."""
    ref, ref_lse, a_abs = refs
    got = hg.bf16_bits_to_f32(out_bits).astype(np.float64)
    err = tol.check_values(got, ref, a_abs, u_p=tol.U_F16 if fp8 else tol.U_BF16, mean=np.inf,
                           label="fp8" if fp8 else "out")
    stats["max"] = max(stats.get("max", 0.0), float(err.max()))
    stats["sum"] = stats.get("sum", 0.0) + float(err.sum())
    stats["n"] = stats.get("n", 0) + err.size
    tol.check_lse(lse, ref_lse)


def _rows(reqs):
    return sorted((r.rid, r.matched, r.first, tuple(int(x) for x in r.slots)) for r in reqs)


def run(trace, runner_fn, pool, cuda, cascade=True, policy=ra.RC_LPM, cache_cls=ra.RadixCache, kv_fp8=False, **kw):
    model = SynthModel(trace.shape, trace.seed, trace.vocab, device=cuda)
    eng = DeviceEngine(trace.shape, pool, device=cuda, kv_fp8=kv_fp8)
    cache = cache_cls(pool)
    log = []
    runner = wl.Runner(cache, model, eng, policy=policy, cascade=cascade, collect=True, log=log,
                       prefill_attention=not trace.shape.mla)
    res = runner_fn(runner, trace, **kw)
    assert ra.rc_sync(eng.err) == ra.RC_OK
    return runner, model, cache, log, res


def check_requests(runner, model, rids, shape, stats, max_decode_steps=None, fp8=False):
    for rid in rids:
        h = model.hashes(rid)
        if rid in runner.extend_out:
            pos, o, l = runner.extend_out[rid]
            compare(o, l, oracle_positions(shape, h, pos, fp8), stats, fp8)
        dec = runner.decode_out.get(rid, [])
        if max_decode_steps is not None:
            dec = [d for i, d in enumerate(dec) if i in max_decode_steps]
        if dec:
            pos = [p for p, _, _ in dec]
            compare(np.stack([o for _, o, _ in dec]), np.stack([l for _, _, l in dec]),
                    oracle_positions(shape, h, pos, fp8), stats, fp8)


def test_tiny_config_all_outputs_vs_oracle(cuda):
    tr = traces.tiny()
    runner, model, cache, log, reqs = run(tr, wl.run_tiny, tr.pool_slots, cuda)
    stats = {}
    check_requests(runner, model, [r.rid for r in reqs], tr.shape, stats)
    assert stats["sum"] / stats["n"] <= MEAN_ABS
    # the same trace through the oracle tree and the oracle's own scheduling
    # round: every request's match, first position and slot row, and the tree
    ot = oracle.OracleTree(tr.pool_slots)
    orunner = wl.Runner(ot, SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu"), sched=oracle.OracleServer(ot))
    oreqs = wl.run_tiny(orunner, tr)
    assert _rows(oreqs) == _rows(reqs)
    assert ot.dump() == cache.dump() and ot.stats() == cache.stats()


def test_few_shot_reduced_cascade_and_flat(cuda):
    tr = traces.few_shot(n_questions=48, max_new=6)
    stats = {}
    outs = {}
    for cascade in (True, False):
        runner, model, cache, log, reqs = run(tr, wl.run_few_shot, 1 << 16, cuda, cascade=cascade)
        if cascade:
            assert runner.last_layout.use_cascade and len(runner.last_layout.segments) == 1
        check_requests(runner, model, [r.rid for r in reqs[::7]], tr.shape, stats)
        outs[cascade] = {rid: np.stack([o for _, o, _ in d]) for rid, d in runner.decode_out.items()}
        assert cache.stats()["match_hit_tokens"] == 48 * len(tr.warm)
    assert stats["sum"] / stats["n"] <= MEAN_ABS
    for rid in outs[True]:
        a = hg.bf16_bits_to_f32(outs[True][rid]).astype(np.float64)
        b = hg.bf16_bits_to_f32(outs[False][rid]).astype(np.float64)
        assert np.abs(a - b).max() <= MAX_ABS


def test_cache_on_equals_cache_off_recompute(cuda):
    """With the cache off every request computes its whole prompt; the outputs
    of the shared-prefix path must agree within the same bound."""
    tr = traces.few_shot(n_questions=24, max_new=4)
    runner_on, *_ = run(tr, wl.run_few_shot, 1 << 15, cuda)

    class NoCache:
        """Every lookup misses: a fresh tree per request."""

        def __init__(self, pool):
            self.pool = pool
            self.inner = ra.RadixCache(pool)

        def __getattr__(self, name):
            return getattr(self.inner, name)

        def match(self, tokens, pin):
            st, m, s, node = self.inner.match(tokens[:0], pin)
            return st, 0, s[:0], node

        def insert(self, tokens, slots, pin):
            st, present, node, canon = self.inner.insert(tokens[:0], slots[:0], pin)
            # keep every slot private: give them back at finish through free()
            return st, 0, node, np.asarray(slots, np.int32)

    model = SynthModel(tr.shape, tr.seed, tr.vocab, device=cuda)
    eng = DeviceEngine(tr.shape, 1 << 17, device=cuda)
    off = wl.Runner(NoCache(1 << 17), model, eng, cascade=False, collect=True)
    wl.run_few_shot(off, tr, warm=False)
    for rid_on, rid_off in zip(sorted(runner_on.decode_out)[:24], sorted(off.decode_out)[:24]):
        a = np.stack([o for _, o, _ in runner_on.decode_out[rid_on]])
        b = np.stack([o for _, o, _ in off.decode_out[rid_off]])
        d = np.abs(hg.bf16_bits_to_f32(a).astype(np.float64) - hg.bf16_bits_to_f32(b))
        assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS


def test_agent_tree_cascade_vs_oracle(cuda):
    tr = traces.agent_tree(root_len=512, branch_len=64, max_new=5)
    runner, model, cache, log, reqs = run(tr, wl.run_agent, 8192, cuda, cascade=True)
    lay = runner.last_layout
    assert lay.use_cascade and len(lay.segments) == 1 + 4 + 16
    stats = {}
    check_requests(runner, model, [r.rid for r in reqs[::9]], tr.shape, stats)
    assert stats["sum"] / stats["n"] <= MEAN_ABS


def test_chat_reduced_with_eviction_vs_oracle(cuda):
    tr = traces.chat(n_sessions=16, n_turns=4, umin=32, umax=128, max_new=8)
    tr.max_batch = 6
    runner, model, cache, log, (served, rounds) = run(tr, wl.run_chat, tr.pool_slots, cuda)
    assert cache.stats()["evicted_nodes"] > 0
    stats = {}
    check_requests(runner, model, [r.rid for r in served[::5]], tr.shape, stats)
    assert stats["sum"] / stats["n"] <= MEAN_ABS


def test_mla_reduced_vs_oracle(cuda):
    """Latent long-context decode: shared prefix + private contexts stored,
    then batched decode; sampled requests against the oracle."""
    tr = traces.mla_long(batch=12, shared_len=512, private_max=1500, steps=3)
    runner, model, cache, log, reqs = run(tr, lambda r, t: wl.run_mla(r, t), tr.pool_slots + 1024, cuda,
                                          cascade=False)
    stats = {}
    check_requests(runner, model, [r.rid for r in reqs[::3]], tr.shape, stats)
    assert stats["sum"] / stats["n"] <= MEAN_ABS
    assert cache.stats()["match_hit_tokens"] >= 12 * 512


@pytest.mark.parametrize("cache_kind", ["radix", "block16"])
def test_multimodal_image_keys_vs_oracle(cuda, cache_kind):
    """Questions about images whose key runs share the tree (or 16-token
    blocks): prefill and decode of sampled requests against the oracle, and the
    host results identical to the oracle cache running the same trace."""
    from oracle import block_oracle as bo
    tr = traces.multimodal(n_images=5, per_image=4, image_tokens=96, max_new=4)
    make = ra.RadixCache if cache_kind == "radix" else (lambda n: ra.BlockCache(n, 16))
    runner, model, cache, log, reqs = run(tr, lambda r, t: wl.run_multimodal(r, t, ra.rc_image_key, batch=4),
                                          tr.pool_slots, cuda, cache_cls=make)
    stats = {}
    check_requests(runner, model, [r.rid for r in reqs[::3]], tr.shape, stats)
    assert stats["sum"] / stats["n"] <= MEAN_ABS
    # later questions about an image reuse its run
    assert cache.stats()["match_hit_tokens"] > len(reqs) * len(tr.system)
    # the oracle cache with the oracle's own scheduling round
    if cache_kind == "radix":
        oc = oracle.OracleTree(tr.pool_slots)
        osched = oracle.OracleServer(oc)
    else:
        oc = bo.OracleBlockCache(tr.pool_slots, 16)
        osched = bo.OracleBlockServer(oc)
    orunner = wl.Runner(oc, SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu"), sched=osched)
    oreqs = wl.run_multimodal(orunner, tr, bo.image_key, batch=4)
    assert _rows(oreqs) == _rows(reqs) and oc.stats() == cache.stats()


@pytest.mark.parametrize("cascade", [True, False])
def test_few_shot_fp8_pool_vs_oracle(cuda, cascade):
    """The few-shot workload (reduced) with an E4M3 pool: prefill over the
    cached examples, decode steps with kv_store quantising each new token;
    sampled requests against the oracle over the oracle's own quantisation of
    the same K/V."""
    tr = traces.few_shot(n_questions=40, max_new=5)
    runner, model, cache, log, reqs = run(tr, wl.run_few_shot, 1 << 16, cuda, cascade=cascade, kv_fp8=True)
    if cascade:
        assert runner.last_layout.use_cascade
    stats = {}
    check_requests(runner, model, [r.rid for r in reqs[::6]], tr.shape, stats, fp8=True)
    assert stats["sum"] / stats["n"] <= MEAN_ABS


def _decode_bits(runner):
    return {rid: np.stack([o for _, o, _ in d]) for rid, d in runner.decode_out.items()}


@pytest.mark.parametrize("which", ["few_shot_batches", "chat"])
def test_overlapped_rounds_equal_serial(cuda, which):
    """The overlapped scheduler (round k's finish and round k+1's admission
    on a worker thread while round k's decode steps are launched) against
    serving round by round: every decode and prefill output bit for bit, and
    the same tree."""
    outs = []
    for overlap in (False, True):
        if which == "chat":
            tr = traces.chat(n_sessions=16, n_turns=4, umin=32, umax=128, max_new=8)
            tr.max_batch = 6
            model = SynthModel(tr.shape, tr.seed, tr.vocab, device=cuda)
            eng = DeviceEngine(tr.shape, tr.pool_slots, device=cuda)
            cache = ra.RadixCache(tr.pool_slots)
            runner = wl.Runner(cache, model, eng, collect=True)
            wl.run_chat(runner, tr, overlap=overlap)
            assert cache.stats()["evicted_nodes"] > 0
        else:
            base = traces.few_shot(n_questions=32, max_new=6)
            model = SynthModel(base.shape, base.seed, base.vocab, device=cuda)
            eng = DeviceEngine(base.shape, 1 << 16, device=cuda)
            cache = ra.RadixCache(1 << 16)
            runner = wl.Runner(cache, model, eng, collect=True)
            runner.serve([runner.request(base.warm, 0)])
            batches = [[runner.request(t.prompt(i), t.max_new) for i in range(32)]
                       for t in (traces.few_shot(n_questions=32, max_new=6, batch_salt=s) for s in range(1, 5))]
            left = list(batches[1:])
            runner.serve_rounds(batches[0], lambda a, w: (left.pop(0) if left else None), None, overlap)
        assert ra.rc_sync(eng.err) == ra.RC_OK
        outs.append((_decode_bits(runner), {k: v[1] for k, v in runner.extend_out.items()}, cache.dump()))
    a, b = outs
    assert a[0].keys() == b[0].keys() and a[1].keys() == b[1].keys() and a[2] == b[2]
    assert all(np.array_equal(a[0][k], b[0][k]) for k in a[0])
    assert all(np.array_equal(a[1][k], b[1][k]) for k in a[1])


@pytest.mark.parametrize("which", ["few_shot_cascade", "few_shot_flat", "few_shot_fp8", "mla"])
def test_decode_runs_equal_single_steps(cuda, which):
    """Runs of decode steps queued by one library call (attn_decode_steps;
    runs of 5 leave ragged ends; inside a run each cascade reads before the
    previous step's table pass ends) against one decode_step call per step:
    every decode output and LSE bit for bit, and the CUDA events the library
    records (one pair per run) cover every step."""
    got = []
    for chunk in (1, 5, 16):
        if which == "mla":
            tr = traces.mla_long(batch=6, shared_len=300, private_max=900, steps=23)
            fn, pool, cascade, fp8 = wl.run_mla, tr.pool_slots, False, False
        else:
            tr = traces.few_shot(n_questions=24, max_new=23)
            fn, pool = wl.run_few_shot, 1 << 16
            cascade, fp8 = which != "few_shot_flat", which == "few_shot_fp8"
        model = SynthModel(tr.shape, tr.seed, tr.vocab, device=cuda)
        eng = DeviceEngine(tr.shape, pool, device=cuda, kv_fp8=fp8)
        runner = wl.Runner(ra.RadixCache(pool), model, eng, cascade=cascade, collect=True,
                           prefill_attention=not tr.shape.mla)
        runner.decode_chunk = chunk
        eng.timing_every = 4
        eng.start_timing(512)
        fn(runner, tr)
        assert ra.rc_sync(eng.err) == ra.RC_OK
        assert runner.last_layout.use_cascade == cascade
        eng.torch.cuda.synchronize()
        evs = eng.events["attn_decode"]
        covered = [t for _, _, info in evs for t in range(info[2], info[2] + (info[3] if len(info) > 3 else 1))]
        # one step in four timed alone; runs timed whole (one pair of events each)
        assert covered == (list(range(0, 23, 4)) if chunk == 1 else list(range(23)))
        assert all(a.elapsed_time(b) > 0 for a, b, _ in evs)
        got.append({rid: (np.stack([o for _, o, _ in d]), np.stack([l for _, _, l in d]))
                    for rid, d in runner.decode_out.items()})
    base = got[0]
    assert len(base) == (6 if which == "mla" else 24)
    for other in got[1:]:
        assert other.keys() == base.keys()
        for rid in base:
            assert np.array_equal(other[rid][0], base[rid][0]) and np.array_equal(other[rid][1], base[rid][1])
