"""Host half of the product library against the oracle, bit for bit.

The same trace of calls runs through both; every returned value (status,
matched length, slot arrays, node ids, eviction logs, orders, statistics)
and the full tree dump must be identical.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import radixattention_prefix_shared_tree_gb300 as ra
from radixattention_prefix_shared_tree_gb300 import workloads as wl
from synth import traces
from synth.model import SynthModel
from tests import scenarios as sc


@pytest.mark.parametrize("seed", range(12))
@pytest.mark.parametrize("vocab,pool", [(3, 24), (5, 64), (50, 200)])
def test_random_traces_bit_exact(built, seed, vocab, pool):
    a, b = oracle.OracleTree(pool), ra.RadixCache(pool)
    la, lb = [], []
    ra_rng, rb_rng = np.random.default_rng(seed), np.random.default_rng(seed)
    sc.random_trace(a, ra_rng, 250, vocab=vocab, log=la)
    sc.random_trace(b, rb_rng, 250, vocab=vocab, log=lb)
    assert len(la) == len(lb)
    for x, y in zip(la, lb):
        assert x == y
    assert a.dump() == b.dump()


def test_dump_after_every_op(built):
    rng = np.random.default_rng(77)
    a, b = oracle.OracleTree(30), ra.RadixCache(30)
    for i in range(200):
        la, lb = [], []
        s = int(rng.integers(0, 1 << 30))
        sc.random_trace(a, np.random.default_rng(s), 1, vocab=3, log=la)
        sc.random_trace(b, np.random.default_rng(s), 1, vocab=3, log=lb)
        assert la == lb
        assert a.dump() == b.dump(), f"op {i}"


@pytest.mark.parametrize("grouped", [False, True])
def test_cyclic_trace_same_log(built, grouped):
    prefixes = traces.cyclic_prefixes(5, 64)
    order = traces.cyclic_order(5, 2, grouped)
    logs = []
    for make in (oracle.OracleTree, ra.RadixCache):
        t = make(256)
        log = []
        for p in order:
            sc.serve_prefill(t, prefixes[p], log)
        logs.append((log, t.dump()))
    assert logs[0] == logs[1]
    hits = sum(1 for e in logs[0][0] if e[1] > 0)
    assert hits == (5 if grouped else 0)


def _host_run(make_cache, trace_fn, runner_fn, seed, vocab, shape, pool, policy=ra.RC_LPM):
    cache = make_cache(pool)
    log = []
    model = SynthModel(shape, seed, vocab, device="cpu")
    runner = wl.Runner(cache, model, engine=None, policy=policy, log=log)
    res = runner_fn(runner, trace_fn())
    return log, cache.dump(), cache.stats(), res


def test_tiny_workload_host_trace(built):
    tr = traces.tiny()
    outs = [_host_run(m, traces.tiny, wl.run_tiny, tr.seed, tr.vocab, tr.shape, tr.pool_slots)
            for m in (oracle.OracleTree, ra.RadixCache)]
    assert outs[0][:3] == outs[1][:3]
    st = outs[1][2]
    # every request after the first finds the 32-token system prompt
    assert st["match_hits"] == len(tr.prompts) - 1


@pytest.mark.parametrize("policy", [ra.RC_LPM, ra.RC_FCFS])
def test_few_shot_workload_host_trace(built, policy):
    small = lambda: traces.few_shot(n_questions=64, max_new=16)
    tr = small()
    outs = [_host_run(m, small, wl.run_few_shot, tr.seed, tr.vocab, tr.shape, 1 << 16, policy)
            for m in (oracle.OracleTree, ra.RadixCache)]
    assert outs[0][:3] == outs[1][:3]
    st = outs[1][2]
    assert st["match_hit_tokens"] == 64 * len(tr.warm)


def test_chat_workload_host_trace_with_eviction(built):
    small = lambda: traces.chat(n_sessions=24, n_turns=5, umin=16, umax=64, max_new=16)
    tr = small()
    tr.max_batch = 8
    outs = []
    for make in (oracle.OracleTree, ra.RadixCache):
        cache = make(tr.pool_slots)
        log = []
        model = SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu")
        runner = wl.Runner(cache, model, log=log)
        served, rounds = wl.run_chat(runner, tr)
        outs.append((log, cache.dump(), cache.stats(), rounds))
    assert outs[0] == outs[1]
    st = outs[1][2]
    assert st["evicted_nodes"] > 0          # the pool holds 75% of the working set
    assert st["match_hits"] > 0


def test_agent_tree_host_trace(built):
    small = lambda: traces.agent_tree(root_len=64, branch_len=8, max_new=8)
    tr = small()
    outs = [_host_run(m, small, wl.run_agent, tr.seed, tr.vocab, tr.shape, 4096)
            for m in (oracle.OracleTree, ra.RadixCache)]
    assert outs[0][:3] == outs[1][:3]


def test_full_chat_host_trace_bit_exact(built):
    """The chat workload at full size (256 sessions x 8 turns, pool = 75% of
    the working set): eviction log, hits and final tree identical."""
    tr = traces.chat()
    outs = []
    for make in (oracle.OracleTree, ra.RadixCache):
        cache = make(tr.pool_slots)
        log = []
        runner = wl.Runner(cache, SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu"), log=log)
        served, rounds = wl.run_chat(runner, tr)
        outs.append((log, cache.stats(), rounds))
    assert outs[0] == outs[1]
    assert outs[1][1]["evicted_tokens"] > 0


def _native_vs_per_call(trace_fn, runner_fn, pool):
    """The scheduler's native batch path (rc_admit / rc_commit) against its
    per-call path (which the tests above pin to the oracle)."""
    out = []
    for log in (None, []):
        tr = trace_fn()
        cache = ra.RadixCache(pool(tr))
        runner = wl.Runner(cache, SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu"), log=log)
        res = runner_fn(runner, tr)
        reqs = res[0] if isinstance(res, tuple) else res
        rows = sorted((r.rid, r.matched, r.first, tuple(int(x) for x in r.slots)) for r in reqs)
        out.append((cache.dump(), cache.stats(), rows))
    assert out[0] == out[1]


def test_native_batch_scheduler_equals_per_call_few_shot(built):
    _native_vs_per_call(lambda: traces.few_shot(n_questions=40, max_new=8), wl.run_few_shot, lambda tr: 1 << 15)


def test_native_batch_scheduler_equals_per_call_chat_with_eviction(built):
    def small():
        tr = traces.chat(n_sessions=20, n_turns=4, umin=16, umax=64, max_new=16)
        tr.max_batch = 7
        return tr
    _native_vs_per_call(small, wl.run_chat, lambda tr: tr.pool_slots)


def test_native_batch_scheduler_equals_per_call_tiny_and_agent(built):
    _native_vs_per_call(traces.tiny, wl.run_tiny, lambda tr: tr.pool_slots)
    _native_vs_per_call(lambda: traces.agent_tree(root_len=64, branch_len=8, max_new=8), wl.run_agent,
                        lambda tr: 4096)


@pytest.mark.parametrize("which", ["few_shot", "agent"])
def test_tree_cascade_plan_equals_slot_row_plan(built, which):
    """rc_cascade_plan (read off the pinned paths of the tree) finds the same
    segments, rows and private starts as the compressed trie of slot rows."""
    from radixattention_prefix_shared_tree_gb300.driver import plan_cascade
    if which == "few_shot":
        tr = traces.few_shot(n_questions=30, max_new=4)
        cache = ra.RadixCache(1 << 15)
        runner = wl.Runner(cache, SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu"))
        runner.serve([runner.request(tr.warm, 0)])
        reqs = [runner.request(tr.prompt(i), tr.max_new) for i in range(30)]
    else:
        tr = traces.agent_tree(root_len=96, branch_len=16, max_new=4)
        cache = ra.RadixCache(8192)
        runner = wl.Runner(cache, SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu"))
        runner.serve([runner.request(tr.root, 0)])
        for lvl in (1, 2):
            runner.serve([runner.request(tr.prompt(p), 0) for p in sorted({lf[:lvl] for lf in tr.leaves})])
        reqs = [runner.request(tr.prompt(lf), tr.max_new) for lf in tr.leaves]
    admitted, _ = runner.sched.admit(reqs)
    runner.sched.commit_prompts(admitted)
    plan = cache.cascade_plan([r.node for r in admitted])
    segs, private = plan_cascade([r.slots[:r.prompt_len] for r in admitted])
    got = set()
    ip, rp = plan["seg_indptr"], plan["seg_row_indptr"]
    for k in range(plan["n_seg"]):
        got.add((tuple(int(x) for x in plan["seg_slots"][ip[k]:ip[k + 1]]),
                 tuple(int(x) for x in plan["seg_rows"][rp[k]:rp[k + 1]])))
    want = {(tuple(int(x) for x in s), tuple(int(x) for x in r)) for s, r in segs}
    assert got == want and len(got) == (1 if which == "few_shot" else 1 + 4 + 16)
    assert (plan["private"] == private).all()
    for b in range(len(admitted)):   # the inverse map lists row b's entries
        pos = plan["req_seg_pos"][plan["req_seg_indptr"][b]:plan["req_seg_indptr"][b + 1]]
        assert all(plan["seg_rows"][p] == b for p in pos)
