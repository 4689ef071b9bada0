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
from radixattention_prefix_shared_tree_gb300.driver import Scheduler
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


class Recorder:
    """Wraps a scheduling object: records every round's admitted requests in
    admission order (rid, matched, first position, pinned node, slot row) and
    the waiting ones, every commit's nodes and slot rows, and the cache's
    statistics (and, with dumps=True, its full dump) after each commit."""

    def __init__(self, sched, cache, dumps=True):
        self.sched, self.cache, self.dumps, self.rec = sched, cache, dumps, []

    def _state(self):
        return self.cache.dump() if self.dumps else tuple(sorted(self.cache.stats().items()))

    def admit(self, pending, policy, max_batch=None):
        a, w = self.sched.admit(pending, policy, max_batch)
        self.rec.append(("admit", [(r.rid, r.matched, r.first, r.node, tuple(int(x) for x in r.slots)) for r in a],
                         sorted(r.rid for r in w)))
        return a, w

    def commit_prompts(self, batch):
        self.sched.commit_prompts(batch)
        self.rec.append(("prefill", [(r.rid, r.node, tuple(int(x) for x in r.slots[:r.prompt_len])) for r in batch],
                         self._state()))

    def finish(self, batch):
        self.sched.finish(batch)
        self.rec.append(("finish", [(r.rid, r.node, tuple(int(x) for x in r.slots)) for r in batch], self._state()))


def _served(kind, trace_fn, runner_fn, pool, policy=ra.RC_LPM, dumps=True):
    """One host run of a workload.  kind: "oracle" (the oracle tree with the
    oracle's own admission round and commits), "native" (the library's
    rc_admit / rc_commit), "per_call" (the driver's per-call scheduler over
    the library's tree)."""
    tr = trace_fn()
    if kind == "oracle":
        cache = oracle.OracleTree(pool(tr))
        inner = oracle.OracleServer(cache)
    else:
        cache = ra.RadixCache(pool(tr))
        inner = Scheduler(cache, None if kind == "native" else [])
    rec = Recorder(inner, cache, dumps)
    runner = wl.Runner(cache, SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu"), policy=policy, sched=rec)
    res = runner_fn(runner, tr)
    return rec.rec, cache.dump(), cache.stats(), res


def _three_way(trace_fn, runner_fn, pool, policy=ra.RC_LPM, dumps=True):
    """The oracle's admission round against the library's native batch path
    and the driver's per-call path: every round's records identical."""
    outs = {k: _served(k, trace_fn, runner_fn, pool, policy, dumps) for k in ("oracle", "native", "per_call")}
    for k in ("native", "per_call"):
        a, b = outs["oracle"], outs[k]
        assert len(a[0]) == len(b[0]), k
        for i, (x, y) in enumerate(zip(a[0], b[0])):
            assert x == y, f"{k}: record {i} ({x[0]}) differs"
        assert a[1] == b[1] and a[2] == b[2], k
    return outs["oracle"]


def test_tiny_workload_host_trace(built):
    tr = traces.tiny()
    rec, dump, st, res = _three_way(traces.tiny, wl.run_tiny, lambda t: t.pool_slots)
    # every request after the first finds the 32-token system prompt
    assert st["match_hits"] == len(tr.prompts) - 1


@pytest.mark.parametrize("policy", [ra.RC_LPM, ra.RC_FCFS])
def test_few_shot_workload_host_trace(built, policy):
    rec, dump, st, res = _three_way(lambda: traces.few_shot(n_questions=64, max_new=16), wl.run_few_shot,
                                    lambda t: 1 << 16, policy)
    assert st["match_hit_tokens"] == 64 * len(traces.few_shot(n_questions=1).warm)


def test_chat_workload_host_trace_with_eviction(built):
    def small():
        tr = traces.chat(n_sessions=24, n_turns=5, umin=16, umax=64, max_new=16)
        tr.max_batch = 8
        return tr
    rec, dump, st, (served, rounds) = _three_way(small, wl.run_chat, lambda t: t.pool_slots)
    assert st["evicted_nodes"] > 0          # the pool holds 75% of the working set
    assert st["match_hits"] > 0
    # some rounds stopped at a request that did not fit (the first misfit rule)
    assert any(r[0] == "admit" and r[2] for r in rec)


def test_chat_admission_misfit_stops_round(built):
    """A pool so small that most rounds end at a misfit after evicting: the
    shortfall eviction and the no-overtaking rule, round by round."""
    def tight():
        tr = traces.chat(n_sessions=12, n_turns=4, umin=40, umax=90, max_new=24)
        tr.pool_slots = 700
        return tr
    rec, dump, st, (served, rounds) = _three_way(tight, wl.run_chat, lambda t: t.pool_slots)
    stops = sum(1 for r in rec if r[0] == "admit" and r[2])
    assert stops >= 3 and st["evicted_nodes"] > 0


def test_agent_tree_host_trace(built):
    _three_way(lambda: traces.agent_tree(root_len=64, branch_len=8, max_new=8), wl.run_agent, lambda t: 4096)


def test_full_chat_host_trace_bit_exact(built):
    """The chat workload at full size (256 sessions x 8 turns, pool = 75% of
    the working set): every round's admissions, slots, evictions (through the
    statistics after each commit) and the final tree identical."""
    rec, dump, st, (served, rounds) = _three_way(traces.chat, wl.run_chat, lambda t: t.pool_slots, dumps=False)
    assert st["evicted_tokens"] > 0 and rounds >= 8


def test_fully_cached_prompt_recomputes_last_token(built):
    """The reading that a request whose whole prompt is cached and that will
    decode recomputes its last prompt token (one new token carries the
    query), while a prefill-only request computes nothing: fixed by hand on
    the oracle's round, then the library's rounds equal it."""
    t = oracle.OracleTree(64)
    srv = oracle.OracleServer(t)

    class R:
        def __init__(self, rid, toks, plen, mnew):
            self.rid, self.tokens, self.prompt_len, self.max_new = rid, np.asarray(toks, np.int32), plen, mnew
            self.node, self.slots = -1, None

    a = R(0, [5, 6, 7, 8], 4, 0)
    adm, _ = srv.admit([a], ra.RC_FCFS)
    assert adm == [a] and (a.matched, a.first) == (0, 0) and list(a.slots) == [0, 1, 2, 3]
    srv.commit_prompts([a])
    b = R(1, [5, 6, 7, 8, 50, 51], 4, 2)       # prompt fully cached, decodes 2
    c = R(2, [5, 6, 7, 8], 4, 0)               # prompt fully cached, prefill only
    adm, _ = srv.admit([b, c], ra.RC_FCFS)
    assert (b.matched, b.first) == (4, 3) and list(b.slots) == [0, 1, 2, 4, 5, 6]
    assert (c.matched, c.first) == (4, 4) and list(c.slots) == [0, 1, 2, 3]
    srv.commit_prompts([b, c])
    assert list(b.slots[:4]) == [0, 1, 2, 3]    # slot 4 duplicated position 3 and was freed
    srv.finish([b, c])
    assert t.stats()["free"] == 64 - 6 and t.stats()["insert_dup_freed"] == 1


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


def test_admission_evicts_shortfall_and_misfit_stops(built):
    """Eviction for room and the first-misfit rule, fixed by hand on the
    oracle's round (note 49, section 4: evict least-recently-used unpinned
    leaves to make room in the shared pool; section 5 serving order), then
    the library's native round must give the same."""
    class R:
        def __init__(self, rid, toks, mnew=0):
            self.rid, self.tokens, self.prompt_len, self.max_new = rid, np.asarray(toks, np.int32), len(toks) - mnew, mnew
            self.node, self.slots = -1, None

    results = []
    for kind in ("oracle", "native"):
        cache = oracle.OracleTree(10) if kind == "oracle" else ra.RadixCache(10)
        srv = oracle.OracleServer(cache) if kind == "oracle" else Scheduler(cache)
        for rid, toks in ((0, [1, 2, 3]), (1, [4, 5, 6, 7])):      # two cached leaves, A older than B
            r = R(rid, toks)
            adm, _ = srv.admit([r], ra.RC_FCFS)
            srv.commit_prompts(adm)
            srv.finish(adm)
        c, d, e = R(2, [9] * 5), R(3, [8] * 6), R(4, [7])
        adm, wait = srv.admit([c, d, e], ra.RC_FCFS)
        results.append(([r.rid for r in adm], [r.rid for r in wait], list(c.slots), cache.stats(), cache.dump()))
    o = results[0]
    # C needs 5 with 3 free: evicts the shortfall (2) = leaf A (3 slots), takes the 5 smallest free ids
    assert o[0] == [2] and o[2] == [0, 1, 2, 7, 8]
    # D needs 6 with 1 free: evicts B (4), still short, no candidate left: unpinned, round ends;
    # E would fit now but does not overtake D
    assert o[1] == [3, 4]
    assert o[3]["evicted_nodes"] == 2 and o[3]["free"] == 5 and o[3]["caller"] == 5 and o[3]["pins"] == 1
    assert results[1] == o


@pytest.mark.parametrize("which", ["chat", "multimodal"])
def test_overlapped_rounds_equal_serial_host(built, which):
    """The overlapped scheduler (round k's finish and round k+1's admission
    on a worker thread) makes the same tree calls in the same order as
    serving round by round: identical records, tree and statistics."""
    outs = []
    for overlap in (False, True):
        if which == "chat":
            tr = traces.chat(n_sessions=20, n_turns=4, umin=16, umax=64, max_new=16)
            tr.max_batch = 7
            run = lambda runner: wl.run_chat(runner, tr, overlap=overlap)
        else:
            tr = traces.multimodal(n_images=4, per_image=5, image_tokens=40, image_bytes=64, max_new=5)
            run = lambda runner: wl.run_multimodal(runner, tr, ra.rc_image_key, batch=3, overlap=overlap)
        cache = ra.RadixCache(tr.pool_slots)
        rec = Recorder(Scheduler(cache), cache)
        run(wl.Runner(cache, SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu"), sched=rec))
        outs.append((rec.rec, cache.dump(), cache.stats()))
    assert outs[0] == outs[1]
    assert any(r[0] == "admit" and r[2] for r in outs[0][0])   # rounds with waiting requests


@pytest.mark.parametrize("seed", range(6))
def test_random_rounds_admit_commit_bit_exact(built, seed):
    """Random multi-round serving against the oracle's own admission round
    and commits (note 49, sections 2, 4 and 5): prompts drawn as extensions
    of earlier ones over a 4-token vocabulary (deep sharing, mid-edge
    splits, fully cached prompts that recompute their last token), a pool
    small enough to evict inside admission, batch caps, prefill-only
    requests.  The native path inserts from each request's pinned node and
    reuses the order's peek lengths; every record, tree and statistic must
    equal the oracle's."""
    class R:
        def __init__(self, rid, toks, mnew):
            self.rid, self.tokens = rid, np.asarray(toks, np.int32)
            self.prompt_len, self.max_new = len(toks) - mnew, mnew
            self.node, self.slots = -1, None

    def run(kind):
        rng = np.random.default_rng(seed)
        cache = oracle.OracleTree(160) if kind == "oracle" else ra.RadixCache(160)
        srv = oracle.OracleServer(cache) if kind == "oracle" else Scheduler(cache)
        seen, rec, rid = [np.asarray([0, 1], np.int32)], [], 0
        pending = []
        for rnd in range(30):
            for _ in range(int(rng.integers(1, 5))):
                base = seen[int(rng.integers(0, len(seen)))]
                cut = int(rng.integers(0, len(base) + 1))
                extra = rng.integers(0, 4, int(rng.integers(0 if cut else 1, 9))).astype(np.int32)
                prompt = np.concatenate([base[:cut], extra]).astype(np.int32)
                if len(prompt) == 0:
                    continue
                mnew = int(rng.integers(0, 4))
                gen = rng.integers(0, 4, mnew).astype(np.int32)
                pending.append(R(rid, np.concatenate([prompt, gen]), mnew))
                seen.append(np.concatenate([prompt, gen]))
                rid += 1
            policy = ra.RC_LPM if rng.random() < 0.8 else ra.RC_FCFS
            cap = int(rng.integers(1, 5)) if rng.random() < 0.5 else None
            adm, wait = srv.admit(pending, policy, cap)
            rec.append(("admit", [(r.rid, r.matched, r.first, tuple(int(x) for x in r.slots)) for r in adm],
                        sorted(r.rid for r in wait)))
            srv.commit_prompts(adm)
            rec.append(("prefill", [(r.rid, tuple(int(x) for x in r.slots[:r.prompt_len])) for r in adm],
                        cache.dump(), sorted(cache.stats().items())))
            srv.finish(adm)
            rec.append(("finish", [(r.rid, tuple(int(x) for x in r.slots)) for r in adm],
                        cache.dump(), sorted(cache.stats().items())))
            pending = wait
        return rec

    a, b = run("oracle"), run("native")
    assert len(a) == len(b)
    for i, (x, y) in enumerate(zip(a, b)):
        assert x == y, f"record {i} ({x[0]}) differs"
    assert any(r[0] == "admit" and r[2] for r in a)                       # rounds left requests waiting
    assert any(dict(r[3])["evicted_nodes"] for r in a if r[0] == "finish")  # admission evicted
