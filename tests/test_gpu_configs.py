"""The five workloads at full size, as the benchmark runs them, against the oracle.

Host results (match lengths, slots, eviction, hit counts, final tree) are
compared bit for bit with the oracle tree replaying the same trace on the
CPU.  Attention outputs are compared on sampled requests and positions, the
oracle recomputing each sampled request's K/V from its own token sequence.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import radixattention_prefix_shared_tree_gb300 as ra
from radixattention_prefix_shared_tree_gb300 import workloads as wl
from radixattention_prefix_shared_tree_gb300.driver import DeviceEngine
from synth import traces
from synth.model import SynthModel
from synth import hashgen as hg
from tests.test_gpu_workloads import MAX_ABS, MEAN_ABS, oracle_positions, compare

pytestmark = pytest.mark.gpu


def _check(runner, model, shape, rids, steps=None):
    stats = {}
    for rid in rids:
        h = model.hashes(rid)
        if rid in runner.extend_out:
            pos, o, l = runner.extend_out[rid]
            pick = np.unique(np.linspace(0, len(pos) - 1, min(len(pos), 24)).astype(int))
            compare(o[pick], l[pick], oracle_positions(shape, h, pos[pick]), stats)
        dec = runner.decode_out.get(rid, [])
        if steps is not None:
            dec = [d for i, d in enumerate(dec) if i in steps]
        if dec:
            compare(np.stack([o for _, o, _ in dec]), np.stack([l for _, _, l in dec]),
                    oracle_positions(shape, h, [p for p, _, _ in dec]), stats)
    assert stats["n"] > 0 and stats["sum"] / stats["n"] <= MEAN_ABS
    return stats


def _gpu_run(tr, fn, pool, cuda, rids, cascade=True):
    model = SynthModel(tr.shape, tr.seed, tr.vocab, device=cuda)
    eng = DeviceEngine(tr.shape, pool, device=cuda)
    cache = ra.RadixCache(pool)
    runner = wl.Runner(cache, model, eng, cascade=cascade, collect=True, prefill_attention=not tr.shape.mla)
    runner.collect_rids = set(rids) if rids is not None else None
    res = fn(runner, tr)
    assert ra.rc_sync(eng.err) == ra.RC_OK
    return runner, model, cache, res


def _oracle_host(tr, fn, pool):
    """The same trace through the oracle tree and the oracle's own
    scheduling round and commits (none of the driver's code)."""
    tree = oracle.OracleTree(pool)
    runner = wl.Runner(tree, SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu"), sched=oracle.OracleServer(tree))
    fn(runner, tr)
    return tree


def _all_decode(runner):
    return {rid: np.stack([o for _, o, _ in d]) for rid, d in runner.decode_out.items()}


def _same_within(a, b, what):
    """Two kernel paths over the same inputs: every output within 1e-2 (both
    are within their bound of the exact value), mean within 1e-3."""
    assert a.keys() == b.keys() and a, what
    worst, tot, n = 0.0, 0.0, 0
    for rid in a:
        d = np.abs(hg.bf16_bits_to_f32(a[rid]).astype(np.float64) - hg.bf16_bits_to_f32(b[rid]))
        worst, tot, n = max(worst, float(d.max())), tot + float(d.sum()), n + d.size
    assert worst <= MAX_ABS and tot / n <= MEAN_ABS, (what, worst, tot / n)


def test_few_shot_full(cuda):
    tr = traces.few_shot()
    rids = {1, 2, 100, 256}
    runner, model, cache, reqs = _gpu_run(tr, wl.run_few_shot, tr.pool_slots, cuda, rids)
    assert runner.last_layout.use_cascade
    _check(runner, model, tr.shape, sorted(rids), steps={0, 1, 64, 127})
    st = cache.stats()
    assert st["match_hit_tokens"] == 256 * len(tr.warm) and st["match_hits"] == 256
    ot = _oracle_host(tr, wl.run_few_shot, tr.pool_slots)
    assert ot.stats() == cache.stats() and ot.dump() == cache.dump()


def test_few_shot_full_cascade_equals_flat(cuda):
    """Every decode output of the full few-shot batch (256 requests x 128
    steps x 32 heads): the cascade path (the shared 1792 keys read once for
    all rows) against the flat path (every row reads its whole context)."""
    tr = traces.few_shot()
    outs = []
    for cascade in (True, False):
        runner, model, cache, reqs = _gpu_run(tr, wl.run_few_shot, tr.pool_slots, cuda, None, cascade=cascade)
        assert runner.last_layout.use_cascade == cascade
        outs.append(_all_decode(runner))
    _same_within(outs[0], outs[1], "few-shot cascade vs flat")


def test_chat_full(cuda):
    """Full chat trace; sampled requests against the oracle, and one whole
    session (its 8 turns) against a cache-disabled recompute: every turn's
    prompt computed from scratch on an empty tree, then the same 128 decode
    steps -- outputs within the bound of the cached path's."""
    tr = traces.chat()
    # which requests are session 5's turns (a host-only run of the same trace)
    hr = wl.Runner(ra.RadixCache(tr.pool_slots), SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu"))
    served_h, _ = wl.run_chat(hr, tr)
    session = sorted((r.rid, r.prompt_len) for r in served_h if r.session == 5)
    rids = {3, 300, 1200, 2040} | {rid for rid, _ in session}
    runner, model, cache, (served, rounds) = _gpu_run(tr, wl.run_chat, tr.pool_slots, cuda, rids)
    assert cache.stats()["evicted_nodes"] > 0 and rounds >= 8
    _check(runner, model, tr.shape, sorted(r for r in {3, 300, 1200, 2040} if r < runner.next_rid),
           steps={0, 127})
    ot = _oracle_host(tr, wl.run_chat, tr.pool_slots)
    assert ot.stats() == cache.stats() and ot.dump() == cache.dump()
    # cache off: each turn alone on an empty tree, its whole prompt prefilled
    by_rid = {r.rid: r for r in served}
    off = {}
    for rid, plen in session:
        r = by_rid[rid]
        eng = DeviceEngine(tr.shape, plen + r.max_new + 64, device=cuda)
        tree = ra.RadixCache(plen + r.max_new + 64)
        offr = wl.Runner(tree, model, eng, cascade=False, collect=True)
        offr.next_rid = rid                # the same request id: same sequence, same hashes
        rr = offr.request(r.prompt, r.max_new)
        admitted, waiting = offr.serve([rr])
        assert admitted and admitted[0].first == 0 and ra.rc_sync(eng.err) == ra.RC_OK
        off[rid] = np.stack([o for _, o, _ in offr.decode_out[rid]])
    on = {rid: np.stack([o for _, o, _ in runner.decode_out[rid]]) for rid, _ in session}
    _same_within(on, off, "chat session cached vs cache-off recompute")


def test_agent_tree_full(cuda):
    tr = traces.agent_tree()
    leaves0 = 1 + 4 + 16
    rids = {leaves0, leaves0 + 37, leaves0 + 63}
    runner, model, cache, reqs = _gpu_run(tr, wl.run_agent, tr.pool_slots, cuda, rids)
    lay = runner.last_layout
    assert lay.use_cascade and len(lay.segments) == 21
    _check(runner, model, tr.shape, sorted(rids), steps={0, 100, 255})
    ot = _oracle_host(tr, wl.run_agent, tr.pool_slots)
    assert ot.stats() == cache.stats() and ot.dump() == cache.dump()


def test_agent_tree_full_cascade_equals_flat(cuda):
    """All 64 leaves x 256 decode steps x 64 heads of the full agent tree:
    the 21-segment cascade against the flat path."""
    tr = traces.agent_tree()
    outs = []
    for cascade in (True, False):
        runner, model, cache, reqs = _gpu_run(tr, wl.run_agent, tr.pool_slots, cuda, None, cascade=cascade)
        assert runner.last_layout.use_cascade == cascade
        outs.append(_all_decode(runner))
    assert len(outs[0]) == 64
    _same_within(outs[0], outs[1], "agent tree cascade vs flat")


def test_mla_full(cuda):
    tr = traces.mla_long()
    lens = [len(p) for p in tr.private]
    # the shortest, a middling and the longest private context (4k to ~32.8k keys)
    order = np.argsort(lens)
    pick = [int(order[0]), int(order[len(order) // 4]), int(order[-1])]
    rids = {1 + i for i in pick}
    runner, model, cache, reqs = _gpu_run(tr, wl.run_mla, tr.pool_slots, cuda, rids, cascade=False)
    _check(runner, model, tr.shape, sorted(rids), steps={0, 63})
    assert cache.stats()["match_hit_tokens"] >= 128 * 4096
    assert max(r.prompt_len for r in reqs) == 4096 + max(lens)
