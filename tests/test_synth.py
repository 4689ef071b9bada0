"""The shared input generator: the C restatement equals the numpy definition,
values have the intended distribution, and identical prefixes give identical rows."""
from __future__ import annotations

import numpy as np

from synth import hashgen as hg
from synth import native, traces


def test_c_hash_scan_equals_numpy(built):
    rng = np.random.default_rng(0)
    tok = rng.integers(0, 32000, 500).astype(np.int32)
    a = hg.prefix_hashes(tok, 1234)
    b = native.prefix_hashes_from(hg.root_hash(1234), tok)
    assert (a == b).all()
    rows = hg.prefix_hashes_rows(tok.reshape(5, 100), np.full(5, hg.root_hash(9), np.uint64))
    for i in range(5):
        assert (rows[i] == hg.prefix_hashes(tok.reshape(5, 100)[i], 9)).all()


def test_c_decode_model_equals_numpy(built):
    h = int(hg.prefix_hashes(np.arange(7, dtype=np.int32), 5)[-1])
    toks, hs = native.decode_tokens(h, 20, 1000)
    state = h
    for i in range(20):
        y = hg.gen_token(state, 1000)
        assert y == toks[i]
        state = int(hg.prefix_hashes_from(state, [y])[0])
        assert state == int(hs[i])


def test_value_distribution():
    h = hg.prefix_hashes(np.arange(4000, dtype=np.int32) % 977, 3)
    v = hg.bf16_bits_to_f32(hg.gen_values(h, hg.KIND_K, 4, 64)).astype(np.float64)
    assert abs(v.mean()) < 0.01 and abs(v.var() - 1.0) < 0.01
    assert np.abs(v).max() <= 6.0


def test_traces_shapes():
    tr = traces.few_shot()
    assert len(tr.warm) == 512 + 5 * 256 and len(tr.questions) == 256
    assert all(32 <= len(q) <= 64 for q in tr.questions)
    assert len({int(q[0]) for q in tr.questions}) == 256
    at = traces.agent_tree()
    assert len(at.leaves) == 64 and len(at.prompt(at.leaves[0])) == 2048 + 3 * 256
    ml = traces.mla_long()
    assert len(ml.private) == 128 and all(0 <= len(p) <= 28672 for p in ml.private)
    ch = traces.chat()
    assert len(ch.user_turns) == 256 and all(len(t) == 8 for t in ch.user_turns)
