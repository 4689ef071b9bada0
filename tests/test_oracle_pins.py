"""Pins of the CPU oracle against what the pages and the mathematics fix.

Nothing here compares the oracle with itself: the tree is pinned by the values
and shapes the pages print (split example, outputs staying cached, the churn
counts, the cyclic sweep, the walkthrough's events), by brute force over all
serving orders (longest-prefix-first optimality, and the size of the trie of a
batch as the lower bound on computed tokens), and by invariants of the rules.
Attention is pinned by closed forms and by torch's own scaled-dot-product
attention in float64.
"""
from __future__ import annotations

import itertools
import os

import numpy as np
import pytest
import torch

import oracle
from synth import traces
from synth.hashgen import KIND_K, KIND_Q, KIND_V, bf16_bits_to_f32, gen_values, prefix_hashes
from tests import scenarios as sc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    rows = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if line and not line.startswith("#"):
            rows.append(line.split())
    return rows


def _nodes(tree):
    out = []
    for line in tree.dump().splitlines():
        head, rest = line.split(":", 1)
        nid, parent, ref, stamp, ntok = (int(x) for x in head.split())
        toks, slots = rest.split("|")
        out.append(dict(id=nid, parent=parent, ref=ref, stamp=stamp, ntok=ntok,
                        tokens=[int(x) for x in toks.split()], slots=[int(x) for x in slots.split()]))
    return out


# ----------------------------------------------------------------- tree pins
def test_split_example_note49_s2(oracle_built):
    """Request 1 = system + Q1 is one path; request 2 = system + Q2 splits the
    edge into a shared part and two branches; only Q2 is computed."""
    sys_p = [11, 12, 13, 14, 15, 16]
    q1, q2 = [21, 22, 23], [31, 32]
    t = oracle.OracleTree(64)
    st, s1 = t.alloc(len(sys_p) + len(q1))
    assert st == 0
    st, present, n1, _ = t.insert(sys_p + q1, s1, False)
    assert (st, present) == (0, 0)
    nodes = _nodes(t)
    assert len(nodes) == 2 and nodes[1]["tokens"] == sys_p + q1  # a single path from the root

    st, m, mslots, node = t.match(sys_p + q2, True)
    assert m == len(sys_p) and list(mslots) == list(s1[:len(sys_p)])
    st, new = t.alloc(len(q2))          # only Q2 needs new KV
    assert len(new) == 2
    st, present, n2, _ = t.insert(sys_p + q2, np.concatenate([mslots, new]), False)
    assert present == len(sys_p)
    assert t.release(node) == 0
    nodes = _nodes(t)
    by_parent = {}
    for n in nodes:
        by_parent.setdefault(n["parent"], []).append(n)
    shared = by_parent[0]
    assert len(shared) == 1 and shared[0]["tokens"] == sys_p          # the shared part
    branches = by_parent[shared[0]["id"]]
    assert sorted(b["tokens"] for b in branches) == sorted([q1, q2])   # two branches
    assert t.stats()["insert_new_tokens"] == len(sys_p) + len(q1) + len(q2)


def test_outputs_stay_cached_note49_s2(oracle_built):
    """A finished turn (prompt and generated answer) is matched whole by the next turn."""
    t = oracle.OracleTree(128)
    turn1 = list(range(100, 120))      # system + user message
    answer = list(range(200, 210))     # generated tokens
    st, s = t.alloc(len(turn1) + len(answer))
    t.insert(turn1 + answer, s, False)
    nxt = turn1 + answer + [300, 301, 302]
    st, m, _, node = t.match(nxt, True)
    assert m == len(turn1) + len(answer)


@pytest.mark.parametrize("row", _golden("churn_note49_s6.txt"))
def test_churn_counts_note49_s6(oracle_built, row):
    n_pref, length, cap, cycles, order, hits, reqs = row
    prefixes = traces.cyclic_prefixes(int(n_pref), int(length))
    seq = traces.cyclic_order(int(n_pref), int(cycles), grouped=(order == "grouped"))
    assert len(seq) == int(reqs)
    got = sc.cyclic_hits(oracle.OracleTree, prefixes, seq, int(cap) * int(length))
    assert got == int(hits)


@pytest.mark.parametrize("row", _golden("sweep_note49_s6.txt"))
def test_cyclic_sweep_note49_s6(oracle_built, row):
    cap, hits, reqs = (int(x) for x in row)
    prefixes = traces.cyclic_prefixes(5, 64)
    seq = traces.cyclic_order(5, 200, grouped=False)
    assert len(seq) == reqs
    assert sc.cyclic_hits(oracle.OracleTree, prefixes, seq, cap * 64) == hits


def _trie_size(prompts):
    root = {}
    size = 0
    for p in prompts:
        node = root
        for tok in p:
            if tok not in node:
                node[tok] = {}
                size += 1
            node = node[tok]
    return size


def _batches(seed, n):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        k = int(rng.integers(3, 7))
        # a few shared stems so that orders matter
        stems = [rng.integers(0, 50, int(rng.integers(1, 6))).astype(np.int32) for _ in range(2)]
        prompts = []
        for _ in range(k):
            stem = stems[int(rng.integers(0, 2))]
            tail = rng.integers(0, 50, int(rng.integers(1, 5))).astype(np.int32)
            prompts.append(np.concatenate([stem, tail]).astype(np.int32))
        out.append(prompts)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_lpm_reaches_bruteforce_optimum_note49_s5(oracle_built, seed):
    """Longest-cached-prefix-first (re-ranked after each request) computes as
    few tokens as the best of all serving orders, when the cache holds at
    least the longest request; the minimum is the size of the batch's trie."""
    for prompts in _batches(seed, 4):
        cap = max(len(p) for p in prompts)
        total = sum(len(p) for p in prompts)
        best = 0
        for perm in itertools.permutations(range(len(prompts))):
            best = max(best, sc.run_batch_sequential(oracle.OracleTree(cap), prompts, perm))
        lpm = sc.lpm_dynamic_order(oracle.OracleTree(cap), prompts)
        assert lpm == best
        assert total - best == _trie_size([tuple(p) for p in prompts])


def test_eviction_rules_note49_s4(oracle_built):
    """Pinned nodes are never evicted; only leaves go; least recently used first;
    a node whose children are gone becomes evictable; the shared trunk goes last."""
    t = oracle.OracleTree(64)
    trunk = [1, 2, 3, 4]
    a, b, c = trunk + [10, 11], trunk + [20, 21], trunk + [30, 31]
    for p in (a, b, c):
        sc.serve_prefill(t, np.asarray(p, np.int32))
    ids = {tuple(n["tokens"]): n["id"] for n in _nodes(t)}
    st, m, _, pinned = t.match(np.asarray(c, np.int32), True)   # c is running: pinned
    # touch a so that b is the least recently used leaf
    t.match(np.asarray(a, np.int32), False)
    st, freed, log = t.evict(2)
    assert list(log) == [ids[(20, 21)]]
    st, freed, log = t.evict(100)          # a's leaf goes; trunk and c are pinned
    assert list(log) == [ids[(10, 11)]]
    assert freed == 2
    assert t.release(pinned) == 0
    st, freed, log = t.evict(100)          # now c's leaf, then the trunk (became a leaf)
    assert list(log) == [ids[(30, 31)], ids[tuple(trunk)]]
    assert t.stats()["free"] == 64


def test_walkthrough_nine_steps_sglang(oracle_built):
    """The nine steps of the RadixAttention walkthrough (unite.ai article on
    SGLang): which nodes appear, split and get evicted at each step."""
    S = list(range(1000, 1016))                 # system prompt
    c1t1 = [1, 2, 3, 4, 5, 6]                   # chat 1, turn 1 (user + answer)
    c1t2 = [7, 8, 9, 10, 11]                    # chat 1, turn 2
    c2t1 = [41, 42, 43, 44, 45]                 # chat 2, turn 1
    c2t2 = [46, 47, 48, 49]                     # chat 2, turn 2
    shots = list(range(2000, 2010))             # few-shot examples
    q = [[3000 + i, 3100 + i] for i in range(3)]
    t = oracle.OracleTree(64)
    ids = lambda: {tuple(n["tokens"]): n["id"] for n in _nodes(t)}

    def serve(prompt):
        log = []
        m = sc.serve_prefill(t, np.asarray(prompt, np.int32), log)
        assert m >= 0
        return m, log[-1][4]

    # step 1: the tree is empty
    assert len(_nodes(t)) == 1
    # step 2: system prompt + first turn go in as one edge to one new node
    serve(S + c1t1)
    assert [n["ntok"] for n in _nodes(t)] == [0, len(S + c1t1)]
    # step 3: the first turn is found and reused; the new turn is a new node
    m, _ = serve(S + c1t1 + c1t2)
    assert m == len(S + c1t1) and len(_nodes(t)) == 3
    # step 4: a new chat session: the step-2 node splits so both share the system prompt
    m, _ = serve(S + c2t1)
    assert m == len(S)
    tops = [n for n in _nodes(t) if n["parent"] == 0]
    assert len(tops) == 1 and tops[0]["tokens"] == S
    # step 5: chat 2 continues under memory pressure (a running batch holds most
    # of the shared pool): one node from step 4 is evicted, the least recently
    # used leaf, chat 1's second turn; the new turn hangs below chat 2's node
    victim = ids()[tuple(c1t2)]
    st, running = t.alloc(t.stats()["free"] - len(c2t2) + 1)
    m, ev = serve(S + c2t1 + c2t2)
    assert m == len(S + c2t1) and list(ev[2]) == [victim]
    assert t.free(running) == 0
    parent_c2t2 = [n["parent"] for n in _nodes(t) if n["tokens"] == c2t2][0]
    assert parent_c2t2 == ids()[tuple(c2t1)]
    # step 6: a few-shot request shares no prefix: a new child of the root
    m, ev = serve(shots + q[0])
    assert m == 0 and ev is None and len([n for n in _nodes(t) if n["parent"] == 0]) == 2
    # step 7: more few-shot requests share the examples: the step-6 node splits
    for qq in q[1:]:
        serve(shots + qq)
    assert len([n for n in _nodes(t) if n["parent"] == ids()[tuple(shots)]]) == 3
    # step 8: chat 1 sends a new message; all of chat 2's nodes are evicted as
    # the least recently used
    chat2 = {ids()[tuple(c2t1)], ids()[tuple(c2t2)]}
    new_msg = list(range(5000, 5000 + t.stats()["free"] + len(c2t1) + len(c2t2)))
    m, ev = serve(S + c1t1 + new_msg)
    assert m == len(S + c1t1)
    assert set(ev[2]) == chat2
    # step 9: more answers are sampled for a question of the few-shot batch;
    # several nodes are evicted to make room
    m, ev = serve(shots + q[1] + [9000, 9001, 9002, 9003, 9004, 9005])
    assert m == len(shots + q[1]) and len(ev[2]) >= 2


def test_fault_paths(oracle_built):
    t = oracle.OracleTree(8)
    assert t.release(12345) == oracle.ERR_STATE           # unknown node
    st, m, _, root = t.match([1, 2], True)
    assert t.release(root) == 0 and t.release(root) == oracle.ERR_STATE  # unpinned
    assert t.alloc(9)[0] == oracle.ERR_NOMEM
    st, s = t.alloc(2)
    assert t.free([s[0], s[0]]) == oracle.ERR_STATE       # repeated slot
    assert t.free([8]) == oracle.ERR_ARG                  # out of range
    assert t.insert([1, 2], [s[0], 5], False)[0] == oracle.ERR_STATE  # slot 5 not held
    assert t.stats()["caller"] == 2                        # nothing changed
    assert t.evict(-1)[0] == oracle.ERR_ARG


def test_slot_conservation_random_traces(oracle_built):
    for seed in range(5):
        t = oracle.OracleTree(40)
        sc.random_trace(t, np.random.default_rng(seed), 300, log=[])
        s = t.stats()
        assert s["free"] + s["caller"] + s["tree_tokens"] == s["pool"]
        nodes = _nodes(t)
        by_id = {n["id"]: n for n in nodes}
        for n in nodes:
            if n["parent"] >= 0:
                assert by_id[n["parent"]]["ref"] >= n["ref"]     # pins cover whole paths
        slots = [x for n in nodes for x in n["slots"]]
        assert len(slots) == len(set(slots))                      # each slot owned once


# ------------------------------------------------------------ attention pins
def _rand_bf16(rng, shape):
    f = rng.standard_normal(shape).astype(np.float32)
    return (torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16))


def test_attention_closed_forms(oracle_built):
    rng = np.random.default_rng(1)
    Hq, Hkv, d = 4, 2, 16
    v = _rand_bf16(rng, (5, Hkv, d))
    k = _rand_bf16(rng, (5, Hkv, d))
    q = _rand_bf16(rng, (1, Hq, d))
    # ctx = 1: the output is the single value row
    out, lse = oracle.attention(q, k, v, [0], [1], Hq, Hkv, d, d, 0.3)
    for h in range(Hq):
        g = h * Hkv // Hq
        np.testing.assert_array_equal(out[0, h], bf16_bits_to_f32(v[0, g]).astype(np.float64))
    # all keys equal: uniform weights, mean of values, lse = s + log(ctx)
    keq = np.repeat(k[:1], 5, axis=0)
    out, lse = oracle.attention(q, keq, v, [0], [5], Hq, Hkv, d, d, 0.3)
    vf = bf16_bits_to_f32(v).astype(np.float64)
    kf = bf16_bits_to_f32(k).astype(np.float64)
    qf = bf16_bits_to_f32(q).astype(np.float64)
    for h in range(Hq):
        g = h * Hkv // Hq
        np.testing.assert_allclose(out[0, h], vf[:, g].mean(0), rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse[0, h], 0.3 * qf[0, h] @ kf[0, g] + np.log(5), rtol=1e-12)
    # q = 0: uniform weights as well
    out, lse = oracle.attention(np.zeros_like(q), k, v, [0], [5], Hq, Hkv, d, d, 0.3)
    np.testing.assert_allclose(out[0, 0], vf[:, 0].mean(0), rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(lse[0], np.log(5), rtol=1e-12)
    # two keys: weights are a logistic function of the score difference
    out, _ = oracle.attention(q, k, v, [0], [2], Hq, Hkv, d, d, 0.3)
    s0, s1 = 0.3 * qf[0, 0] @ kf[0, 0], 0.3 * qf[0, 0] @ kf[1, 0]
    w0 = 1.0 / (1.0 + np.exp(s1 - s0))
    np.testing.assert_allclose(out[0, 0], w0 * vf[0, 0] + (1 - w0) * vf[1, 0], rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("Hq,Hkv,d", [(4, 4, 64), (32, 8, 128), (8, 1, 32)])
def test_attention_matches_torch_sdpa_prefill(oracle_built, Hq, Hkv, d):
    """Causal prefill of n new tokens over a cached prefix P (keys 0..P+i for
    new token i) against torch's scaled_dot_product_attention in float64."""
    rng = np.random.default_rng(Hq + d)
    P, n = 23, 9
    k = _rand_bf16(rng, (P + n, Hkv, d))
    v = _rand_bf16(rng, (P + n, Hkv, d))
    q = _rand_bf16(rng, (n, Hq, d))
    scale = 1.0 / np.sqrt(d)
    out, lse = oracle.attention(q, k, v, np.zeros(n, np.int64), P + np.arange(n) + 1, Hq, Hkv, d, d, scale)
    kt = torch.from_numpy(bf16_bits_to_f32(k)).double().permute(1, 0, 2)   # [Hkv, T, d]
    vt = torch.from_numpy(bf16_bits_to_f32(v)).double().permute(1, 0, 2)
    qt = torch.from_numpy(bf16_bits_to_f32(q)).double().permute(1, 0, 2)   # [Hq, n, d]
    G = Hq // Hkv
    kt, vt = kt.repeat_interleave(G, 0), vt.repeat_interleave(G, 0)
    mask = torch.arange(P + n)[None, :] <= (P + torch.arange(n))[:, None]
    ref = torch.nn.functional.scaled_dot_product_attention(qt[None], kt[None], vt[None], attn_mask=mask[None, None],
                                                           scale=scale)[0]
    np.testing.assert_allclose(out, ref.permute(1, 0, 2).numpy(), rtol=1e-10, atol=1e-12)


def test_attention_latent_matches_sdpa(oracle_built):
    """One latent KV head (576 wide), V = its first 512 columns, 16 query heads."""
    rng = np.random.default_rng(7)
    T, Hq = 40, 16
    k = _rand_bf16(rng, (T, 1, 576))
    q = _rand_bf16(rng, (1, Hq, 576))
    scale = 1.0 / np.sqrt(576)
    out, lse = oracle.attention(q, k, None, [0], [T], Hq, 1, 576, 512, scale, latent=True)
    kf = torch.from_numpy(bf16_bits_to_f32(k)).double()[:, 0]
    qf = torch.from_numpy(bf16_bits_to_f32(q)).double()[0]
    ref = torch.nn.functional.scaled_dot_product_attention(qf[None, :, None, :], kf[None, None].expand(1, Hq, T, 576),
                                                           kf[None, None, :, :512].expand(1, Hq, T, 512), scale=scale)
    np.testing.assert_allclose(out[0], ref[0, :, 0].numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(lse[0], torch.logsumexp(scale * qf @ kf.T, dim=1).numpy(), rtol=1e-12)


def test_attention_key_order_invariance(oracle_built):
    rng = np.random.default_rng(3)
    k = _rand_bf16(rng, (12, 2, 32))
    v = _rand_bf16(rng, (12, 2, 32))
    q = _rand_bf16(rng, (1, 4, 32))
    perm = rng.permutation(12)
    a, la = oracle.attention(q, k, v, [0], [12], 4, 2, 32, 32, 0.2)
    b, lb = oracle.attention(q, k[perm], v[perm], [0], [12], 4, 2, 32, 32, 0.2)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(la, lb, rtol=1e-12)


def test_prefix_hash_inputs_make_reuse_exact(oracle_built):
    """Identical prefixes give identical K/V: cached rows equal recomputed rows."""
    a = np.asarray([5, 6, 7, 8, 9], np.int32)
    b = np.asarray([5, 6, 7, 1, 2], np.int32)
    ha, hb = prefix_hashes(a, 99), prefix_hashes(b, 99)
    assert (ha[:3] == hb[:3]).all() and (ha[3:] != hb[3:]).all()
    for kind in (KIND_K, KIND_V, KIND_Q):
        va, vb = gen_values(ha, kind, 2, 8), gen_values(hb, kind, 2, 8)
        assert (va[:3] == vb[:3]).all()
