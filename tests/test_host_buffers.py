"""Host-side buffer reuse in the scheduler: a round's slot rows live in one
flat array that a later round may take again only once no request refers to
it, and every admitted row must still equal the oracle's admission round
(note 49, sections 4 and 5: match, pin, allocate from the shared pool)."""
from __future__ import annotations

import gc

import numpy as np

import oracle
import radixattention_prefix_shared_tree_gb300 as ra
from radixattention_prefix_shared_tree_gb300.driver import Request, Scheduler


def _requests(rng, base, n, rid0):
    out = []
    for i in range(n):
        tail = rng.integers(0, 1000, int(rng.integers(3, 9))).astype(np.int32)
        gen = rng.integers(0, 1000, 4).astype(np.int32)
        toks = np.concatenate([base, tail, gen]).astype(np.int32)
        out.append(Request(rid=rid0 + i, tokens=toks, prompt_len=len(base) + len(tail), max_new=4))
    return out


def _twin(reqs):
    return [Request(rid=r.rid, tokens=r.tokens.copy(), prompt_len=r.prompt_len, max_new=r.max_new) for r in reqs]


def _round(nat, orc, reqs):
    a, wa = nat.admit(reqs, ra.RC_LPM)
    twins = _twin(reqs)
    b, wb = orc.admit(twins, ra.RC_LPM)
    assert not wa and not wb
    assert [r.rid for r in a] == [r.rid for r in b]
    for x, y in zip(a, b):
        assert (x.matched, x.first) == (y.matched, y.first)
        assert np.array_equal(x.slots, y.slots)
    return a, b


def test_row_buffers_reused_only_when_unreferenced(built):
    rng = np.random.default_rng(5)
    base = rng.integers(0, 1000, 24).astype(np.int32)
    nat = Scheduler(ra.RadixCache(4096))
    orc = oracle.OracleServer(oracle.OracleTree(4096))

    # batch A's requests kept alive: batch B's admission must not write into their rows
    a1, b1 = _round(nat, orc, _requests(rng, base, 6, 0))
    addr1 = a1[0].slots.__array_interface__["data"][0]
    for s in (nat, orc):
        s.commit_prompts(a1 if s is nat else b1)
        s.finish(a1 if s is nat else b1)
    kept = [r.slots.copy() for r in a1]      # after the commits (they write canonical slots)
    a2, b2 = _round(nat, orc, _requests(rng, base, 6, 100))
    assert all(np.array_equal(r.slots, k) for r, k in zip(a1, kept))
    assert not np.shares_memory(a1[0].slots, a2[0].slots)
    for s in (nat, orc):
        s.commit_prompts(a2 if s is nat else b2)
        s.finish(a2 if s is nat else b2)

    # batch A's requests dropped: batch C's admission takes A's buffer again, rows still exact
    del a1, b1, kept
    gc.collect()
    a3, b3 = _round(nat, orc, _requests(rng, base, 6, 200))
    starts = {r.slots.__array_interface__["data"][0] for r in a3}
    assert min(starts) == addr1
    for s in (nat, orc):
        s.commit_prompts(a3 if s is nat else b3)
        s.finish(a3 if s is nat else b3)
    assert nat.cache.dump() == orc.cache.dump()


def test_row_buffer_pool_is_bounded(built):
    rng = np.random.default_rng(6)
    base = rng.integers(0, 1000, 16).astype(np.int32)
    nat = Scheduler(ra.RadixCache(1 << 14))
    held = []
    for k in range(Scheduler.ROW_BUFFERS + 3):   # every batch's requests kept alive
        a, _ = nat.admit(_requests(rng, base, 4, 10 * k), ra.RC_LPM)
        nat.commit_prompts(a)
        nat.finish(a)
        held.append(a)
    assert len(nat._rows) <= Scheduler.ROW_BUFFERS
    rows = [r.slots for a in held for r in a]
    for i in range(len(rows)):          # no two live rows overlap
        for j in range(i + 1, len(rows)):
            assert not np.shares_memory(rows[i], rows[j])


def test_tokens_addr_follows_the_array():
    r = Request(rid=0, tokens=np.arange(10, dtype=np.int64), prompt_len=6, max_new=4)
    p = r.tokens_addr()
    assert r.tokens.dtype == np.int32 and r.tokens.flags.c_contiguous
    assert p == r.tokens.ctypes.data and r.tokens_addr() == p
    r.tokens = np.arange(20, 30, dtype=np.int32)
    assert r.tokens_addr() == r.tokens.ctypes.data != p
    v = np.arange(40, dtype=np.int32)[::2]        # strided: copied once
    r.tokens = v
    q = r.tokens_addr()
    assert r.tokens is not v and r.tokens.flags.c_contiguous and q == r.tokens.ctypes.data
    assert np.array_equal(r.tokens, v)
