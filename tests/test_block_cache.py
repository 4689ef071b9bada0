"""The block-granular comparator cache and image keys (CPU).

Oracle pins: the closed form of reuse against shared-prefix length that the
note's vLLM comparison (section 3) draws -- whole 16-token blocks vs every
token -- the churn counts and the cyclic sweep of its section 6, equality with
the separately pinned radix-tree oracle where the two schemes must agree, and
the published FNV-1a / splitmix64 values behind image keys.  Then the product
against the oracle, result by result.
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import radixattention_prefix_shared_tree_gb300 as ra
from oracle import block_oracle as bo
from radixattention_prefix_shared_tree_gb300 import workloads as wl
from synth import traces
from synth.model import SynthModel
from tests import scenarios as sc


def serve(cache, prompt):
    """One prefill-only request alone; frees the partial last block."""
    st, m, ms, node = cache.match(prompt, True)
    assert st == 0
    st, new = cache.alloc(len(prompt) - m)
    assert st == 0
    slots = np.concatenate([ms, new]).astype(np.int32)
    st, present, node2, canon = cache.insert(prompt, slots, False)
    assert st == 0 and present == m
    assert cache.release(node) == 0
    k = cache.uncached_tail(len(prompt)) if hasattr(cache, "uncached_tail") else 0
    if k:
        assert cache.free(canon[len(prompt) - k:]) == 0
    return m


# ----------------------------------------------------------------- oracle pins
@pytest.mark.parametrize("L", list(range(0, 81, 1)))
def test_reuse_vs_shared_prefix_length(L):
    """Note 49 s.3: blocks are matched whole (16 tokens), the radix tree down to
    the token: a second prompt sharing L tokens reuses 16*floor(L/16) vs L."""
    rng = np.random.default_rng(L)
    a = rng.integers(0, 1000, 96).astype(np.int32)
    b = np.concatenate([a[:L], [1000 + L], rng.integers(0, 1000, 20)]).astype(np.int32)
    blk, rad = bo.OracleBlockCache(1024, 16), oracle.OracleTree(1024)
    serve(blk, a)
    serve(rad, a)
    assert blk.match(b, False)[1] == 16 * (L // 16)
    assert rad.match(b, False)[1] == L


@pytest.mark.parametrize("grouped,hits", [(False, 0), (True, 5)])
def test_churn_counts_block_granular(grouped, hits):
    """Note 49 s.6 with 64-token prefixes (four whole blocks) and a cache of
    four prefixes: cycling A..E twice finds nothing, pairs find 5 of 10."""
    prefixes = traces.cyclic_prefixes(5, 64)
    order = traces.cyclic_order(5, 2, grouped)
    assert sc.cyclic_hits(lambda n: bo.OracleBlockCache(n, 16), prefixes, order, 256) == hits


@pytest.mark.parametrize("k", range(1, 7))
def test_cyclic_sweep_block_granular(k):
    """Note 49 s.6: no hit until the cache holds the working set, then every
    request after the first cycle hits (995 of 1000)."""
    prefixes = traces.cyclic_prefixes(5, 64)
    order = traces.cyclic_order(5, 200, False)
    hits = sc.cyclic_hits(lambda n: bo.OracleBlockCache(n, 16), prefixes, order, 64 * k)
    assert hits == (0 if k < 5 else 995)


def _block_words(rng, n_words, B, vocab_words):
    """Prompts made of whole B-token words whose first tokens differ, so two
    prompts can only share a multiple of B tokens."""
    words = [np.concatenate([[w], rng.integers(1000, 2000, B - 1)]).astype(np.int32) for w in range(vocab_words)]
    return [np.concatenate([words[int(i)] for i in rng.integers(0, vocab_words, int(rng.integers(1, n_words + 1)))])
            for _ in range(40)]


@pytest.mark.parametrize("seed", range(4))
def test_block_aligned_traces_match_radix(seed):
    """Where every shared prefix is a whole number of blocks and nothing is
    evicted, block and radix matching reuse exactly the same tokens."""
    rng = np.random.default_rng(seed)
    prompts = _block_words(rng, 6, 16, 3)
    blk, rad = bo.OracleBlockCache(1 << 14, 16), oracle.OracleTree(1 << 14)
    for p in prompts:
        assert serve(blk, p) == serve(rad, p)


@pytest.mark.parametrize("seed", range(4))
def test_one_token_blocks_match_radix(seed):
    """Blocks of one token are a trie of single tokens: the same matches as the
    radix tree on any trace without eviction."""
    rng = np.random.default_rng(100 + seed)
    blk, rad = bo.OracleBlockCache(1 << 12, 1), oracle.OracleTree(1 << 12)
    for _ in range(60):
        p = rng.integers(0, 3, int(rng.integers(1, 14))).astype(np.int32)
        assert serve(blk, p) == serve(rad, p)


def test_eviction_invariants_under_pressure():
    """Pinned blocks and the root are never evicted; a chain shrinks from its
    end (no evicted block leaves a live child behind); slots are conserved."""
    rng = np.random.default_rng(5)
    c = bo.OracleBlockCache(48, 4)
    pins = []
    for _ in range(400):
        p = rng.integers(0, 3, int(rng.integers(1, 17))).astype(np.int32)
        st, m, ms, node = c.match(p, True)
        st, new = c.alloc(len(p) - m)
        if st != 0:
            before = {b.id for b in c.blocks.values()}
            pinned = {b.id for b in c.blocks.values() if b.ref > 0}
            est, freed, log = c.evict(len(p) - m - c.stats()["free"])
            assert 0 not in log and not (set(int(x) for x in log) & pinned)
            gone = set(int(x) for x in log)
            assert all(b.parent not in gone for b in c.blocks.values() if b.id in before)
            st, new = c.alloc(len(p) - m)
        if st != 0:
            assert c.release(node) == 0
            continue
        slots = np.concatenate([ms, new]).astype(np.int32)
        st, present, node2, canon = c.insert(p, slots, True)
        assert st == 0
        assert c.release(node) == 0
        pins.append((node2, canon, len(p)))
        if len(pins) > 3 or rng.random() < 0.5:
            n2, cn, n = pins.pop(0)
            assert c.release(n2) == 0
            k = c.uncached_tail(n)
            if k:
                assert c.free(cn[n - k:]) == 0
        s = c.stats()
        assert s["free"] + s["caller"] + s["tree_tokens"] == 48


def test_image_key_oracle_published_values():
    # FNV-1a 64 of "", "a", "foobar" (the FNV authors' test values)
    assert bo.fnv1a64(b"") == 0xCBF29CE484222325
    assert bo.fnv1a64(b"a") == 0xAF63DC4C8601EC8C
    assert bo.fnv1a64(b"foobar") == 0x85944171F73967E8
    # splitmix64 seeded with 0: its first output is the finaliser of the gamma
    assert bo.splitmix64_finalise(0x9E3779B97F4A7C15) == 0xE220A8397B1DCDAF
    k = bo.image_key(b"picture", 600)
    assert len(k) == 600 and all(-(1 << 30) <= x <= -1 for x in k)
    assert k == bo.image_key(b"picture", 600)
    assert bo.image_key(b"picturf", 600)[0] != k[0]
    assert bo.image_key(b"", 3) == [-1 - (bo.splitmix64_finalise(0xCBF29CE484222325 + i * 0x9E3779B97F4A7C15) >> 34)
                                    for i in (1, 2, 3)]


def test_image_run_is_a_shared_prefix_in_the_tree(built):
    """An image's keys behave as tokens of the tree: the same image matches
    through its run, a different image stops the match where the run starts."""
    sysp = np.arange(10, 40, dtype=np.int32)
    img_a, img_b = b"\x01" * 100, b"\x01" * 99 + b"\x02"
    q1, q2 = np.array([5, 6, 7], np.int32), np.array([8, 9], np.int32)
    for key in (bo.image_key, ra.rc_image_key):
        t = oracle.OracleTree(4096)
        serve(t, np.concatenate([sysp, np.asarray(key(img_a, 64), np.int32), q1]))
        assert t.match(np.concatenate([sysp, np.asarray(key(img_a, 64), np.int32), q2]), False)[1] == 30 + 64
        assert t.match(np.concatenate([sysp, np.asarray(key(img_b, 64), np.int32), q2]), False)[1] == 30


# ------------------------------------------------------ product against oracle
@pytest.mark.parametrize("n", [0, 1, 5, 64, 577])
def test_image_key_product_matches_oracle(built, n):
    rng = np.random.default_rng(n)
    for size in (0, 1, 7, 100, 4096):
        data = rng.integers(0, 256, size, dtype=np.int64).astype(np.uint8).tobytes()
        assert ra.rc_image_key(data, n).tolist() == bo.image_key(data, n)


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("B,vocab,pool", [(4, 3, 24), (4, 5, 64), (2, 50, 200), (16, 2, 128)])
def test_random_traces_bit_exact(built, seed, B, vocab, pool):
    la, lb = [], []
    bases = [np.random.default_rng(1000 + i).integers(0, vocab, 3 * B + 3).astype(np.int32) for i in range(3)]
    sc.random_trace(bo.OracleBlockCache(pool, B), np.random.default_rng(seed), 250, vocab=vocab,
                    max_len=3 * B + 3, log=la, bases=bases)
    sc.random_trace(ra.BlockCache(pool, B), np.random.default_rng(seed), 250, vocab=vocab,
                    max_len=3 * B + 3, log=lb, bases=bases)
    assert la == lb
    # the trace exercised what it should: hits, evictions, duplicates
    assert sum(1 for e in la if e[0] == "match" and e[2] > 0) >= 10
    assert any(e[0] == "evict" and e[2] > 0 for e in la)


def test_workload_host_trace_bit_exact(built):
    """The multimodal workload (small): the oracle block cache served by the
    oracle's own scheduling round (OracleBlockServer) against the product
    block cache under the driver's scheduler; every admitted request's
    matched length, first position and slot row, and the final statistics,
    equal."""
    from radixattention_prefix_shared_tree_gb300.driver import Scheduler
    tr = traces.multimodal(n_images=4, per_image=4, image_tokens=40, image_bytes=64, max_new=5)
    outs = []
    for oracle_side in (True, False):
        cache = bo.OracleBlockCache(tr.pool_slots, 16) if oracle_side else ra.BlockCache(tr.pool_slots, 16)
        sched = bo.OracleBlockServer(cache) if oracle_side else Scheduler(cache, [])
        runner = wl.Runner(cache, SynthModel(tr.shape, tr.seed, tr.vocab, device="cpu"), engine=None, sched=sched)
        served = wl.run_multimodal(runner, tr, bo.image_key if oracle_side else ra.rc_image_key, batch=3)
        outs.append(([(r.rid, r.matched, r.first, tuple(int(x) for x in r.slots)) for r in served],
                     runner.cache.stats()))
    assert outs[0] == outs[1]
    st = outs[1][1]
    assert st["caller"] == 0  # every partial block went back
    assert st["match_hit_tokens"] > 0 and st["evicted_nodes"] >= 0


def test_host_api_errors(built):
    c = ra.BlockCache(16, 4)
    assert c.alloc(17)[0] == ra.RC_ERR_NOMEM
    assert c.release(999) == ra.RC_ERR_STATE
    assert c.release(0) == ra.RC_ERR_STATE
    assert c.free([16]) == ra.RC_ERR_ARG
    assert c.sched_order(7, [[1]])[0] == ra.RC_ERR_ARG
    assert c.evict(-3)[0] == ra.RC_ERR_ARG
    st, s = c.alloc(4)
    assert c.insert([1, 2, 3, 4], [s[0], s[0], s[1], s[2]], False)[0] == ra.RC_ERR_STATE
    assert c.stats()["caller"] == 4 and c.stats()["tree_tokens"] == 0
    with pytest.raises(ra.RCError):
        ra.BlockCache(16, 0)
