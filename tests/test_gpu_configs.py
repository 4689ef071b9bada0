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
from tests.test_gpu_workloads import MEAN_ABS, oracle_positions, compare

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
    runner.collect_rids = set(rids)
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


def test_chat_full(cuda):
    tr = traces.chat()
    rids = {3, 300, 1200, 2040}
    runner, model, cache, (served, rounds) = _gpu_run(tr, wl.run_chat, tr.pool_slots, cuda, rids)
    assert cache.stats()["evicted_nodes"] > 0 and rounds >= 8
    _check(runner, model, tr.shape, sorted(r for r in rids if r < runner.next_rid), steps={0, 127})
    ot = _oracle_host(tr, wl.run_chat, tr.pool_slots)
    assert ot.stats() == cache.stats() and ot.dump() == cache.dump()


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


def test_mla_full(cuda):
    tr = traces.mla_long()
    lens = [len(p) for p in tr.private]
    # the requests with the shortest and a middling private context (the oracle is O(ctx) per query)
    order = np.argsort(lens)
    pick = [int(order[0]), int(order[len(order) // 4])]
    rids = {1 + i for i in pick}
    runner, model, cache, reqs = _gpu_run(tr, wl.run_mla, tr.pool_slots, cuda, rids, cascade=False)
    _check(runner, model, tr.shape, sorted(rids), steps={0, 63})
    assert cache.stats()["match_hit_tokens"] >= 128 * 4096
