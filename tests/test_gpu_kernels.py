"""CUDA kernels through the C-ABI against the oracle, element by element.

Sizes span several 64-key tiles and split chunks with ragged tails; slot
tables are random permutations of the pool so every gather is scattered.
Bar (attention): |gpu - oracle| <= max(1e-2, the bound the kernels'
arithmetic forces) element by element (``tests/tolerance.py`` derives it:
P's rounding to bf16 before P.V, fp32 slack, and half an ulp of the bf16
output), mean |gpu - oracle| <= 1e-3, |lse - oracle lse| <= 2e-3.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import radixattention_prefix_shared_tree_gb300 as ra
from radixattention_prefix_shared_tree_gb300.driver import plan_cascade
from synth import hashgen as hg
from synth import native
from tests import tolerance as tol

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS, LSE_ABS = tol.MAX_ABS, tol.MEAN_ABS, tol.LSE_ABS


def bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def rand_bf16(gen, shape, dev):
    return torch.randn(*shape, generator=gen, dtype=torch.float32).to(torch.bfloat16).to(dev)


def check(out_bits, refs, lse=None, u_p=tol.U_BF16, label="out"):
    """refs = (exact output, exact lse, A = attention with |V|) from the
    oracle; the output bound is tolerance.bound, the mean bound 1e-3."""
    ref, ref_lse, a_abs = refs
    tol.check_values(hg.bf16_bits_to_f32(out_bits), ref, a_abs, u_p=u_p, label=label)
    if lse is not None:
        tol.check_lse(lse, ref_lse)


class Pool:
    def __init__(self, n_slots, Hkv, D, dev, seed):
        g = torch.Generator().manual_seed(seed)
        self.k = rand_bf16(g, (n_slots, Hkv, D), dev)
        self.v = rand_bf16(g, (n_slots, Hkv, D), dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.desc = ra.make_pool_desc(self.k, self.v, self.err)
        self.kb, self.vb = bits(self.k), bits(self.v)


def test_synth_gpu_generator_equals_numpy(cuda):
    h = hg.prefix_hashes(np.arange(300, dtype=np.int32) * 7 % 1000, 11)
    dh = torch.from_numpy(h.view(np.int64)).to(cuda)
    for kind, heads, dims in ((hg.KIND_K, 8, 128), (hg.KIND_Q, 32, 128), (hg.KIND_K, 1, 576)):
        out = torch.empty(len(h), heads * dims, dtype=torch.bfloat16, device=cuda)
        native.gen_values_gpu(dh, kind, heads, dims, out)
        ref = hg.gen_values(h, kind, heads, dims).reshape(len(h), -1)
        assert (bits(out) == ref).all()


def test_kv_store_scatter_and_append(cuda):
    n_slots, Hkv, D = 500, 8, 128
    pool = Pool(n_slots, Hkv, D, cuda, 0)
    g = torch.Generator().manual_seed(1)
    n = 77
    slots = torch.randperm(n_slots, generator=g)[:n].to(torch.int32).to(cuda)
    k = rand_bf16(g, (n, Hkv, D), cuda)
    v = rand_bf16(g, (n, Hkv, D), cuda)
    table = torch.full((300,), -1, dtype=torch.int32, device=cuda)
    pos = torch.randperm(300, generator=g)[:n].to(torch.int32).to(cuda)
    ra.kv_store(pool.desc, slots, k, v, table, pos)
    assert ra.rc_sync(pool.err) == ra.RC_OK
    s = slots.long()
    assert torch.equal(pool.k[s], k) and torch.equal(pool.v[s], v)
    assert torch.equal(table[pos.long()], slots)
    # a slot outside the pool is skipped and reported; the rest is written
    bad = slots.clone()
    bad[3] = n_slots + 5
    k2 = rand_bf16(g, (n, Hkv, D), cuda)
    ra.kv_store(pool.desc, bad, k2, v)
    assert ra.rc_sync(pool.err) == ra.RC_ERR_DEVICE
    assert torch.equal(pool.k[s[:3]], k2[:3]) and torch.equal(pool.k[s[3]], k[3])
    assert ra.rc_sync(pool.err) == ra.RC_OK   # the error word was cleared


def _tables(lens, n_slots, seed, dev):
    rng = np.random.default_rng(seed)
    rows = [rng.choice(n_slots, size=L, replace=False).astype(np.int32) for L in lens]
    starts = np.zeros(len(lens), np.int64)
    starts[1:] = np.cumsum(lens)[:-1]
    flat = np.concatenate(rows)
    t = torch.from_numpy(flat).to(dev)
    st = torch.from_numpy(starts.astype(np.int32)).to(dev)
    ln = torch.from_numpy(np.asarray(lens, np.int32)).to(dev)
    return rows, t, st, ln


def _oracle_rows(pool, rows, q_bits, ctx_of_row, Hq, Hkv, D, scale):
    """Oracle over gathered K/V: query row i sees the first ctx_of_row[i] keys
    of rows[i].  Returns (out, lse, A) with A the same attention over |V|."""
    ks = np.concatenate([pool.kb[r] for r in rows])
    vs = np.concatenate([pool.vb[r] for r in rows])
    offs = np.zeros(len(rows), np.int64)
    offs[1:] = np.cumsum([len(r) for r in rows])[:-1]
    ctx = np.asarray(ctx_of_row, np.int64)
    out, lse = oracle.attention(q_bits, ks, vs, offs, ctx, Hq, Hkv, D, D, scale)
    a_abs, _ = oracle.attention(q_bits, ks, tol.abs_bits(vs), offs, ctx, Hq, Hkv, D, D, scale)
    return out, lse, a_abs


DECODE_CASES = [
    # Hq, Hkv, D, lens
    (4, 4, 64, [1, 2, 63, 64, 65, 130]),
    (32, 8, 128, [1, 17, 64, 200, 1000, 2500, 4097]),
    (64, 8, 128, [5, 129, 3000]),
    (16, 8, 128, [700, 33]),
    (8, 8, 128, [1, 1024]),
]


@pytest.mark.parametrize("Hq,Hkv,D,lens", DECODE_CASES)
def test_decode_flat_vs_oracle(cuda, Hq, Hkv, D, lens):
    n_slots = 6000
    pool = Pool(n_slots, Hkv, D, cuda, Hq + D)
    rows, table, start, length = _tables(lens, n_slots, 3, cuda)
    g = torch.Generator().manual_seed(2)
    B = len(lens)
    q = rand_bf16(g, (B, Hq, D), cuda)
    scale = 1.0 / np.sqrt(D)
    desc = ra.make_attn_desc(pool.desc, Hq, scale)
    kv = ra.make_kv_table(table, start, length, max(lens))
    ws = torch.empty(ra.attn_decode_workspace(desc, B, max(lens)), dtype=torch.uint8, device=cuda)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=cuda)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda)
    ra.attn_decode(desc, q, kv, B, out, lse, ws)
    assert ra.rc_sync(pool.err) == ra.RC_OK
    refs = _oracle_rows(pool, rows, bits(q), lens, Hq, Hkv, D, scale)
    check(bits(out), refs, lse.cpu().numpy())


EXTEND_CASES = [
    # Hq, Hkv, D, (prefix, new) per request
    (4, 4, 64, [(0, 1), (32, 9), (0, 70), (5, 64)]),
    (32, 8, 128, [(1792, 40), (0, 17), (100, 130), (1792, 64), (0, 1)]),
    (64, 8, 128, [(2048, 33), (300, 8), (0, 200)]),
    (16, 8, 128, [(63, 65)]),
]


@pytest.mark.parametrize("Hq,Hkv,D,reqs", EXTEND_CASES)
def test_extend_vs_oracle(cuda, Hq, Hkv, D, reqs):
    n_slots = 8000
    pool = Pool(n_slots, Hkv, D, cuda, 7 * Hq + D)
    lens = [p + n for p, n in reqs]
    rows, table, start, length = _tables(lens, n_slots, 5, cuda)
    g = torch.Generator().manual_seed(4)
    ns = [n for _, n in reqs]
    T = sum(ns)
    q = rand_bf16(g, (T, Hq, D), cuda)
    qo = torch.tensor(np.concatenate([[0], np.cumsum(ns)]).astype(np.int32), device=cuda)
    scale = 1.0 / np.sqrt(D)
    desc = ra.make_attn_desc(pool.desc, Hq, scale)
    kv = ra.make_kv_table(table, start, length, max(lens))
    out = torch.empty(T, Hq, D, dtype=torch.bfloat16, device=cuda)
    lse = torch.empty(T, Hq, dtype=torch.float32, device=cuda)
    ra.attn_extend(desc, q, qo, kv, len(reqs), max(ns), out, lse)
    assert ra.rc_sync(pool.err) == ra.RC_OK
    row_of, ctx = [], []
    for b, (p, n) in enumerate(reqs):
        for i in range(n):
            row_of.append(rows[b])
            ctx.append(p + i + 1)
    refs = _oracle_rows(pool, row_of, bits(q), ctx, Hq, Hkv, D, scale)
    check(bits(out), refs, lse.cpu().numpy())


@pytest.mark.parametrize("Hq,Hkv,D", [(32, 8, 128), (64, 8, 128), (4, 4, 64)])
def test_cascade_equals_flat_and_oracle(cuda, Hq, Hkv, D):
    """A tree of shared prefixes: root shared by all rows, two mid segments,
    private tails; cascade decode == flat decode == oracle."""
    n_slots = 20000
    pool = Pool(n_slots, Hkv, D, cuda, 99 + Hq)
    rng = np.random.default_rng(8)
    perm = rng.permutation(n_slots).astype(np.int32)
    root, mids = perm[:700], [perm[700:900], perm[900:1157]]
    off = 1157
    rows = []
    for b in range(12):
        tail_len = int(rng.integers(1, 150))
        tail = perm[off:off + tail_len]
        off += tail_len
        mid = mids[b % 2] if b < 10 else np.zeros(0, np.int32)
        rows.append(np.concatenate([root, mid, tail]).astype(np.int32))
    B = len(rows)
    lens = [len(r) for r in rows]
    _, table, start, length = _tables(lens, n_slots, 0, cuda)
    table.copy_(torch.from_numpy(np.concatenate(rows)).to(cuda))
    g = torch.Generator().manual_seed(6)
    q = rand_bf16(g, (B, Hq, D), cuda)
    scale = 1.0 / np.sqrt(D)
    desc = ra.make_attn_desc(pool.desc, Hq, scale)
    # flat
    kv = ra.make_kv_table(table, start, length, max(lens))
    ws = torch.empty(ra.attn_decode_workspace(desc, B, max(lens)), dtype=torch.uint8, device=cuda)
    flat = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=cuda)
    flat_lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda)
    ra.attn_decode(desc, q, kv, B, flat, flat_lse, ws)
    # cascade from the shared structure of the rows (tails are private)
    prefix_rows = [r[:len(r) - 1] for r in rows]
    segs, private = plan_cascade(prefix_rows)
    assert len(segs) == 3
    seg_slots = np.concatenate([s for s, _ in segs]).astype(np.int32)
    seg_indptr = np.concatenate([[0], np.cumsum([len(s) for s, _ in segs])]).astype(np.int32)
    seg_rows = np.concatenate([np.asarray(r, np.int32) for _, r in segs])
    seg_row_indptr = np.concatenate([[0], np.cumsum([len(r) for _, r in segs])]).astype(np.int32)
    pos_of = [[p for p, b in enumerate(seg_rows) if b == bb] for bb in range(B)]
    req_indptr = np.concatenate([[0], np.cumsum([len(x) for x in pos_of])]).astype(np.int32)
    req_pos = np.concatenate([np.asarray(x, np.int32) for x in pos_of])
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(cuda)
    arrs = [T(seg_slots), T(seg_indptr), T(seg_row_indptr), T(seg_rows), T(req_indptr), T(req_pos)]
    casc = ra.make_cascade(*arrs, max_seg_rows=max(len(r) for _, r in segs),
                           max_seg_len=max(len(x) for x, _ in segs))
    pstart = T(start.cpu().numpy() + private)
    plen = T(np.asarray(lens) - private)
    kv2 = ra.make_kv_table(table, pstart, plen, int((np.asarray(lens) - private).max()))
    ws2 = torch.empty(ra.attn_decode_workspace(desc, B, kv2.max_len, casc), dtype=torch.uint8, device=cuda)
    cout = torch.empty_like(flat)
    clse = torch.empty_like(flat_lse)
    ra.attn_decode(desc, q, kv2, B, cout, clse, ws2, cascade=casc)
    # the same cascade with host copies of the segment offsets: a grid of the
    # non-empty (segment, key chunk, row block) items only, the partials of
    # the chunks past a short segment marked empty by its first chunk's CTA;
    # every CTA does the same work as before, so the results are bit-identical
    casc_c = ra.make_cascade(*arrs, max_seg_rows=max(len(r) for _, r in segs),
                             max_seg_len=max(len(x) for x, _ in segs), host_seg_indptr=seg_indptr,
                             host_seg_row_indptr=seg_row_indptr)
    cout_c = torch.empty_like(flat)
    clse_c = torch.empty_like(flat_lse)
    ra.attn_decode(desc, q, kv2, B, cout_c, clse_c, ws2, cascade=casc_c)
    assert ra.rc_sync(pool.err) == ra.RC_OK
    assert (bits(cout_c) == bits(cout)).all()
    assert (clse_c.cpu().numpy().view(np.uint32) == clse.cpu().numpy().view(np.uint32)).all()
    refs = _oracle_rows(pool, rows, bits(q), lens, Hq, Hkv, D, scale)
    check(bits(flat), refs, flat_lse.cpu().numpy(), label="flat")
    check(bits(cout), refs, clse.cpu().numpy(), label="cascade")
    d = np.abs(hg.bf16_bits_to_f32(bits(cout)).astype(np.float64) - hg.bf16_bits_to_f32(bits(flat)))
    assert d.max() <= MAX_ABS and d.mean() <= MEAN_ABS


def _append_vs_store_then_decode(cuda, Hq, Hkv, D, rows, casc_of=None):
    """attn_decode_append on one copy of the pool == kv_store + attn_decode on
    another: outputs and LSE bit for bit, and the pools equal afterwards; the
    result also matches the oracle over the stored pool."""
    n_slots = 20000
    B = len(rows)
    lens = [len(r) for r in rows]
    pa = Pool(n_slots, Hkv, D, cuda, 7 + Hq)
    pb = Pool(n_slots, Hkv, D, cuda, 7 + Hq)
    _, table, start, length = _tables(lens, n_slots, 0, cuda)
    table.copy_(torch.from_numpy(np.concatenate(rows)).to(cuda))
    g = torch.Generator().manual_seed(21)
    q = rand_bf16(g, (B, Hq, D), cuda)
    k_new = rand_bf16(g, (B, Hkv, D), cuda)
    v_new = rand_bf16(g, (B, Hkv, D), cuda)
    last = torch.from_numpy(np.asarray([r[-1] for r in rows], np.int32)).to(cuda)
    scale = 1.0 / np.sqrt(D)
    if casc_of is None:
        kv, casc = ra.make_kv_table(table, start, length, max(lens)), None
    else:
        kv, casc = casc_of(table, start, lens)
    outs = []
    for pool, fused in ((pa, False), (pb, True)):
        desc = ra.make_attn_desc(pool.desc, Hq, scale)
        ws = torch.empty(ra.attn_decode_workspace(desc, B, kv.max_len, casc), dtype=torch.uint8, device=cuda)
        out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=cuda)
        lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda)
        if fused:
            ra.attn_decode_append(desc, q, k_new, v_new, kv, B, out, lse, ws, cascade=casc)
        else:
            ra.kv_store(pool.desc, last, k_new, v_new)
            ra.attn_decode(desc, q, kv, B, out, lse, ws, cascade=casc)
        assert ra.rc_sync(pool.err) == ra.RC_OK
        outs.append((bits(out), lse.cpu().numpy()))
    assert (outs[0][0] == outs[1][0]).all()
    assert (outs[0][1].view(np.uint32) == outs[1][1].view(np.uint32)).all()
    assert (bits(pa.k) == bits(pb.k)).all() and (bits(pa.v) == bits(pb.v)).all()
    pa.kb, pa.vb = bits(pa.k), bits(pa.v)
    refs = _oracle_rows(pa, rows, bits(q), lens, Hq, Hkv, D, scale)
    check(outs[1][0], refs, outs[1][1])


@pytest.mark.parametrize("Hq,Hkv,D,lens", [(32, 8, 128, [1, 17, 64, 200, 3000, 4097]),
                                            (4, 4, 64, [1, 2, 63, 64, 65, 130])])
def test_decode_append_split_rows(cuda, Hq, Hkv, D, lens):
    """Few rows: the keys are split over chunks, the last key sits in the last."""
    rng = np.random.default_rng(5)
    perm = rng.permutation(20000).astype(np.int32)
    offs = np.concatenate([[0], np.cumsum(lens)])
    rows = [perm[offs[i]:offs[i + 1]] for i in range(len(lens))]
    _append_vs_store_then_decode(cuda, Hq, Hkv, D, rows)


def test_decode_append_fused_rows(cuda):
    """Enough rows for one warp per row and KV head (fused epilogue)."""
    rng = np.random.default_rng(6)
    lens = rng.integers(1, 90, size=200)
    perm = rng.permutation(20000).astype(np.int32)
    offs = np.concatenate([[0], np.cumsum(lens)])
    rows = [perm[offs[i]:offs[i + 1]] for i in range(len(lens))]
    _append_vs_store_then_decode(cuda, 32, 8, 128, rows)


def test_decode_append_with_cascade(cuda):
    """Shared root and mid segments in a cascade; the appended key is private."""
    rng = np.random.default_rng(9)
    perm = rng.permutation(20000).astype(np.int32)
    root, mids = perm[:700], [perm[700:900], perm[900:1157]]
    off, rows = 1157, []
    for b in range(12):
        n = int(rng.integers(1, 150))
        rows.append(np.concatenate([root, mids[b % 2] if b < 10 else np.zeros(0, np.int32),
                                    perm[off:off + n]]).astype(np.int32))
        off += n

    def casc_of(table, start, lens):
        segs, private = plan_cascade([r[:len(r) - 1] for r in rows])
        B = len(rows)
        seg_rows = np.concatenate([np.asarray(r, np.int32) for _, r in segs])
        pos_of = [[p for p, b in enumerate(seg_rows) if b == bb] for bb in range(B)]
        T = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(cuda)
        arrs = [T(np.concatenate([s for s, _ in segs])), T(np.concatenate([[0], np.cumsum([len(s) for s, _ in segs])])),
                T(np.concatenate([[0], np.cumsum([len(r) for _, r in segs])])), T(seg_rows),
                T(np.concatenate([[0], np.cumsum([len(x) for x in pos_of])])),
                T(np.concatenate([np.asarray(x, np.int32) for x in pos_of]))]
        casc = ra.make_cascade(*arrs, max_seg_rows=max(len(r) for _, r in segs),
                               max_seg_len=max(len(x) for x, _ in segs))
        plen = np.asarray(lens) - private
        kv = ra.make_kv_table(table, T(start.cpu().numpy() + private), T(plen), int(plen.max()))
        kv._keep = kv._keep + (arrs,)
        return kv, casc

    _append_vs_store_then_decode(cuda, 32, 8, 128, rows, casc_of)


def test_decode_reports_len_above_max_len(cuda):
    """A row longer than the promised max_len is reported, not read past."""
    pool = Pool(300, 8, 128, cuda, 1)
    rows, table, start, length = _tables([200, 250], 300, 1, cuda)
    q = rand_bf16(torch.Generator().manual_seed(0), (2, 32, 128), cuda)
    desc = ra.make_attn_desc(pool.desc, 32, 0.088)
    kv = ra.make_kv_table(table, start, length, 100)
    ws = torch.empty(ra.attn_decode_workspace(desc, 2, 100), dtype=torch.uint8, device=cuda)
    out = torch.empty(2, 32, 128, dtype=torch.bfloat16, device=cuda)
    ra.attn_decode(desc, q, kv, 2, out, None, ws)
    assert ra.rc_sync(pool.err) == ra.RC_ERR_DEVICE


def test_cascade_fused_path_with_empty_tails(cuda):
    """Enough rows that each (row, KV head) is one CTA (merge fused into it);
    some rows have every key in shared segments (empty private part)."""
    Hq, Hkv, D = 32, 8, 128
    n_slots = 30000
    pool = Pool(n_slots, Hkv, D, cuda, 5)
    rng = np.random.default_rng(21)
    perm = rng.permutation(n_slots).astype(np.int32)
    root = perm[:1500]
    mids = [perm[1500:1700], perm[1700:1990]]
    off = 1990
    rows, private = [], []
    B = 48
    for b in range(B):
        mid = mids[b % 2]
        tail_len = 0 if b % 5 == 0 else int(rng.integers(1, 200))
        tail = perm[off:off + tail_len]
        off += tail_len
        rows.append(np.concatenate([root, mid, tail]).astype(np.int32))
        private.append(len(root) + len(mid))
    lens = [len(r) for r in rows]
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(cuda)
    starts = np.concatenate([[0], np.cumsum(lens)[:-1]])
    table = T(np.concatenate(rows))
    segs = [(root, list(range(B))), (mids[0], list(range(0, B, 2))), (mids[1], list(range(1, B, 2)))]
    seg_rows = np.concatenate([np.asarray(r, np.int32) for _, r in segs])
    pos_of = [[p for p, b in enumerate(seg_rows) if b == bb] for bb in range(B)]
    arrs = [T(np.concatenate([s for s, _ in segs])), T(np.concatenate([[0], np.cumsum([len(s) for s, _ in segs])])),
            T(np.concatenate([[0], np.cumsum([len(r) for _, r in segs])])), T(seg_rows),
            T(np.concatenate([[0], np.cumsum([len(x) for x in pos_of])])), T(np.concatenate(pos_of))]
    casc = ra.make_cascade(*arrs, max_seg_rows=B, max_seg_len=len(root))
    private = np.asarray(private)
    plen = np.asarray(lens) - private
    kv = ra.make_kv_table(table, T(starts + private), T(plen), int(plen.max()))
    g = torch.Generator().manual_seed(9)
    q = rand_bf16(g, (B, Hq, D), cuda)
    desc = ra.make_attn_desc(pool.desc, Hq, 1.0 / np.sqrt(D))
    ws = torch.empty(ra.attn_decode_workspace(desc, B, kv.max_len, casc), dtype=torch.uint8, device=cuda)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=cuda)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda)
    ra.attn_decode(desc, q, kv, B, out, lse, ws, cascade=casc)
    assert ra.rc_sync(pool.err) == ra.RC_OK
    refs = _oracle_rows(pool, rows, bits(q), lens, Hq, Hkv, D, 1.0 / np.sqrt(D))
    check(bits(out), refs, lse.cpu().numpy())


@pytest.mark.parametrize("lens", [[1, 31, 33, 700], [5000, 64, 1025], [3] * 40 + [2049] * 8])
def test_decode_latent_vs_oracle(cuda, lens):
    """One 576-wide latent KV head (V = its first 512 columns), 128 query heads:
    single-chunk (fused) and split-chunk (merge) plans."""
    n_slots = 12000
    g = torch.Generator().manual_seed(len(lens))
    pool = rand_bf16(g, (n_slots, 576), cuda)
    err = torch.zeros(1, dtype=torch.int32, device=cuda)
    pd = ra.make_pool_desc(pool, None, err, mla=True, head_dim_v=512)
    B, Hq = len(lens), 128
    rows, table, start, length = _tables(lens, n_slots, 11, cuda)
    q = rand_bf16(g, (B, Hq, 576), cuda)
    scale = 1.0 / np.sqrt(576)
    desc = ra.make_attn_desc(pd, Hq, scale)
    kv = ra.make_kv_table(table, start, length, max(lens))
    ws = torch.empty(ra.attn_decode_workspace(desc, B, max(lens)), dtype=torch.uint8, device=cuda)
    out = torch.empty(B, Hq, 512, dtype=torch.bfloat16, device=cuda)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda)
    ra.attn_decode(desc, q, kv, B, out, lse, ws)
    assert ra.rc_sync(err) == ra.RC_OK
    pb = bits(pool)
    ks = np.concatenate([pb[r] for r in rows])[:, None, :]
    offs = np.concatenate([[0], np.cumsum(lens)[:-1]])
    ref, ref_lse = oracle.attention(bits(q), ks, None, offs, np.asarray(lens), Hq, 1, 576, 512, scale, latent=True)
    # A: the same scores, |V| = |first 512 columns|
    a_abs, _ = oracle.attention(bits(q), ks, tol.abs_bits(ks[:, :, :512]), offs, np.asarray(lens), Hq, 1, 576, 512,
                                scale)
    check(bits(out), (ref, ref_lse, a_abs), lse.cpu().numpy())


# ------------------------------------------------------------------ FP8 pool
class Fp8Pool:
    """An E4M3 pool filled through kv_store (which quantises) from random bf16 rows."""

    def __init__(self, n_slots, Hkv, dev, seed, magnitudes=True):
        g = torch.Generator().manual_seed(seed)
        D = 128
        k = rand_bf16(g, (n_slots, Hkv, D), dev)
        v = rand_bf16(g, (n_slots, Hkv, D), dev)
        if magnitudes:  # rows of very different size, a few all-zero and tiny ones
            k = (k.float() * torch.exp(2 * torch.randn(n_slots, Hkv, 1, generator=g)).to(dev)).to(torch.bfloat16)
            # (values near unit size keep the outputs O(1), where the mean bound means something)
            v = (v.float() * torch.exp(0.5 * torch.randn(n_slots, Hkv, 1, generator=g)).to(dev)).to(torch.bfloat16)
            k[::97] = 0
            v[5::89] = 0
            k[3::101] *= 1e-30
        self.kb, self.vb = bits(k), bits(v)
        self.k8 = torch.zeros(n_slots, Hkv, D, dtype=torch.uint8, device=dev)
        self.v8 = torch.zeros(n_slots, Hkv, D, dtype=torch.uint8, device=dev)
        self.ks = torch.full((n_slots, Hkv), -1.0, dtype=torch.float32, device=dev)
        self.vs = torch.full((n_slots, Hkv), -1.0, dtype=torch.float32, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.desc = ra.make_pool_desc(self.k8, self.v8, self.err, k_scale=self.ks, v_scale=self.vs)
        slots = torch.randperm(n_slots, generator=g).to(torch.int32).to(dev)
        ra.kv_store(self.desc, slots, k[slots.long()].contiguous(), v[slots.long()].contiguous())
        assert ra.rc_sync(self.err) == ra.RC_OK


def test_kv_store_fp8_quantisation_bit_exact(cuda):
    from oracle import fp8_oracle as f8
    pool = Fp8Pool(3000, 8, cuda, 11)
    for codes, scales, src in ((pool.k8, pool.ks, pool.kb), (pool.v8, pool.vs, pool.vb)):
        c_ref, s_ref = f8.quantize_rows(src)
        got_c = codes.cpu().numpy()
        got_s = scales.cpu().numpy()
        assert np.array_equal(got_s.view(np.uint32), s_ref.view(np.uint32))
        # codes equal; the sign of a zero is not compared
        strip = lambda c: np.where((c & 0x7F) == 0, 0, c)
        assert np.array_equal(strip(got_c), strip(c_ref))
    assert (pool.ks.cpu().numpy() == 0).sum() >= 3000 * 8 // 97 - 8


FP8_DECODE_CASES = [
    # Hq, Hkv, lens, rows of very different magnitude
    (32, 8, [1, 17, 64, 200, 1000, 2500, 4097], False),
    (64, 8, [5, 129, 3000], False),
    (8, 8, [1, 1024, 33], False),
    (32, 8, [48 + (i * 37) % 150 for i in range(160)], False),   # one wave, fused epilogue
    (32, 8, [1, 17, 64, 200, 1000, 2500, 4097], True),
]


@pytest.mark.parametrize("Hq,Hkv,lens,magnitudes", FP8_DECODE_CASES)
def test_decode_fp8_flat_vs_oracle(cuda, Hq, Hkv, lens, magnitudes):
    """Against the oracle on the dequantised pool.  Unit-scale rows take the
    usual bar; rows spread over e^(+-8) in size (peaked softmax, outputs up to
    several units) take the same elementwise bound and a mean bound scaled by
    the outputs' size (the bf16 rounding of an output grows with it)."""
    from oracle import fp8_oracle as f8
    n_slots = 24000
    pool = Fp8Pool(n_slots, Hkv, cuda, Hq + len(lens), magnitudes=magnitudes)
    rows, table, start, length = _tables(lens, n_slots, 3, cuda)
    g = torch.Generator().manual_seed(2)
    B = len(lens)
    D = 128
    q = rand_bf16(g, (B, Hq, D), cuda)
    scale = 1.0 / np.sqrt(D)
    desc = ra.make_attn_desc(pool.desc, Hq, scale)
    kv = ra.make_kv_table(table, start, length, max(lens))
    ws = torch.empty(ra.attn_decode_workspace(desc, B, max(lens)), dtype=torch.uint8, device=cuda)
    out = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=cuda)
    lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda)
    ra.attn_decode(desc, q, kv, B, out, lse, ws)
    assert ra.rc_sync(pool.err) == ra.RC_OK
    kd = f8.dequantize(pool.k8.cpu().numpy(), pool.ks.cpu().numpy())
    vd = f8.dequantize(pool.v8.cpu().numpy(), pool.vs.cpu().numpy())
    sel = np.concatenate(rows)
    offs = np.zeros(B, np.int64)
    offs[1:] = np.cumsum(lens)[:-1]
    ref, ref_lse = f8.attention(bits(q), kd[sel], vd[sel], offs, np.asarray(lens), Hq, Hkv, scale)
    a_abs, _ = f8.attention(bits(q), kd[sel], np.abs(vd[sel]), offs, np.asarray(lens), Hq, Hkv, scale)
    if not magnitudes:
        check(bits(out), (ref, ref_lse, a_abs), lse.cpu().numpy(), u_p=tol.U_F16)
        return
    # Outputs of several units: the elementwise bound as everywhere; the mean
    # bound adds the mean rounding of a correctly rounded bf16 output (a
    # quarter ulp on average), which alone exceeds 1e-3 once |o| > ~0.5; the
    # LSE bound grows with the scores' size (fp32 sums of d products).
    got = hg.bf16_bits_to_f32(bits(out)).astype(np.float64)
    tol.check_values(got, ref, a_abs, u_p=tol.U_F16, mean=MEAN_ABS + tol.bf16_ulp(ref).mean() / 4,
                     label="magnitudes")
    tol.check_lse(lse.cpu().numpy(), ref_lse, LSE_ABS * max(1.0, np.abs(ref_lse).max() / 100))


def test_fp8_pool_rejected_where_unsupported(cuda):
    pool = Fp8Pool(512, 8, cuda, 1, magnitudes=False)
    desc = ra.make_attn_desc(pool.desc, 32, 0.1)
    lens = [10, 20]
    rows, table, start, length = _tables(lens, 512, 3, cuda)
    kv = ra.make_kv_table(table, start, length, 20)
    q = torch.zeros(2, 32, 128, dtype=torch.bfloat16, device=cuda)
    out = torch.empty_like(q)
    ws = torch.empty(1 << 20, dtype=torch.uint8, device=cuda)
    kv_new = torch.zeros(2, 8, 128, dtype=torch.bfloat16, device=cuda)
    with pytest.raises(ra.RCError) as e:
        ra.attn_decode_append(desc, q, kv_new, kv_new, kv, 2, out, None, ws)
    assert e.value.status == ra.RC_ERR_UNSUPPORTED


def _fp8_oracle_rows(pool, rows, q_bits, ctx_of_row, Hq, Hkv, scale):
    """The FP8 oracle over gathered rows of the dequantised pool: (out, lse, A)."""
    from oracle import fp8_oracle as f8
    if not hasattr(pool, "kd"):
        pool.kd = f8.dequantize(pool.k8.cpu().numpy(), pool.ks.cpu().numpy())
        pool.vd = f8.dequantize(pool.v8.cpu().numpy(), pool.vs.cpu().numpy())
    sel = np.concatenate(rows)
    offs = np.zeros(len(rows), np.int64)
    offs[1:] = np.cumsum([len(r) for r in rows])[:-1]
    ctx = np.asarray(ctx_of_row, np.int64)
    out, lse = f8.attention(q_bits, pool.kd[sel], pool.vd[sel], offs, ctx, Hq, Hkv, scale)
    a_abs, _ = f8.attention(q_bits, pool.kd[sel], np.abs(pool.vd[sel]), offs, ctx, Hq, Hkv, scale)
    return out, lse, a_abs


@pytest.mark.parametrize("Hq,Hkv,reqs", [
    (32, 8, [(1792, 40), (0, 17), (100, 130), (1792, 64), (0, 1)]),
    (64, 8, [(2048, 33), (300, 8), (0, 200)]),
    (16, 8, [(63, 65)]),
])
def test_extend_fp8_vs_oracle(cuda, Hq, Hkv, reqs):
    n_slots = 8000
    pool = Fp8Pool(n_slots, Hkv, cuda, 7 * Hq, magnitudes=False)
    lens = [p + n for p, n in reqs]
    rows, table, start, length = _tables(lens, n_slots, 5, cuda)
    g = torch.Generator().manual_seed(4)
    ns = [n for _, n in reqs]
    T = sum(ns)
    D = 128
    q = rand_bf16(g, (T, Hq, D), cuda)
    qo = torch.tensor(np.concatenate([[0], np.cumsum(ns)]).astype(np.int32), device=cuda)
    scale = 1.0 / np.sqrt(D)
    desc = ra.make_attn_desc(pool.desc, Hq, scale)
    kv = ra.make_kv_table(table, start, length, max(lens))
    out = torch.empty(T, Hq, D, dtype=torch.bfloat16, device=cuda)
    lse = torch.empty(T, Hq, dtype=torch.float32, device=cuda)
    ra.attn_extend(desc, q, qo, kv, len(reqs), max(ns), out, lse)
    assert ra.rc_sync(pool.err) == ra.RC_OK
    row_of, ctx = [], []
    for b, (p, n) in enumerate(reqs):
        for i in range(n):
            row_of.append(rows[b])
            ctx.append(p + i + 1)
    refs = _fp8_oracle_rows(pool, row_of, bits(q), ctx, Hq, Hkv, scale)
    check(bits(out), refs, lse.cpu().numpy(), u_p=tol.U_F16)


@pytest.mark.parametrize("Hq,Hkv", [(32, 8), (64, 8)])
def test_cascade_fp8_equals_flat_and_oracle(cuda, Hq, Hkv):
    """FP8 pool: cascade decode == flat decode == the FP8 oracle."""
    n_slots, D = 20000, 128
    pool = Fp8Pool(n_slots, Hkv, cuda, 99 + Hq, magnitudes=False)
    rng = np.random.default_rng(8)
    perm = rng.permutation(n_slots).astype(np.int32)
    root, mids = perm[:700], [perm[700:900], perm[900:1157]]
    off = 1157
    rows = []
    for b in range(40):
        tail_len = int(rng.integers(1, 150))
        tail = perm[off:off + tail_len]
        off += tail_len
        mid = mids[b % 2] if b < 30 else np.zeros(0, np.int32)
        rows.append(np.concatenate([root, mid, tail]).astype(np.int32))
    B = len(rows)
    lens = [len(r) for r in rows]
    _, table, start, length = _tables(lens, n_slots, 0, cuda)
    table.copy_(torch.from_numpy(np.concatenate(rows)).to(cuda))
    g = torch.Generator().manual_seed(6)
    q = rand_bf16(g, (B, Hq, D), cuda)
    scale = 1.0 / np.sqrt(D)
    desc = ra.make_attn_desc(pool.desc, Hq, scale)
    kv = ra.make_kv_table(table, start, length, max(lens))
    ws = torch.empty(ra.attn_decode_workspace(desc, B, max(lens)), dtype=torch.uint8, device=cuda)
    flat = torch.empty(B, Hq, D, dtype=torch.bfloat16, device=cuda)
    flat_lse = torch.empty(B, Hq, dtype=torch.float32, device=cuda)
    ra.attn_decode(desc, q, kv, B, flat, flat_lse, ws)
    prefix_rows = [r[:len(r) - 1] for r in rows]
    segs, private = plan_cascade(prefix_rows)
    assert len(segs) == 3
    seg_slots = np.concatenate([s for s, _ in segs]).astype(np.int32)
    seg_indptr = np.concatenate([[0], np.cumsum([len(s) for s, _ in segs])]).astype(np.int32)
    seg_rows = np.concatenate([np.asarray(r, np.int32) for _, r in segs])
    seg_row_indptr = np.concatenate([[0], np.cumsum([len(r) for _, r in segs])]).astype(np.int32)
    pos_of = [[p for p, b in enumerate(seg_rows) if b == bb] for bb in range(B)]
    req_indptr = np.concatenate([[0], np.cumsum([len(x) for x in pos_of])]).astype(np.int32)
    req_pos = np.concatenate([np.asarray(x, np.int32) for x in pos_of])
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(cuda)
    arrs = [T(seg_slots), T(seg_indptr), T(seg_row_indptr), T(seg_rows), T(req_indptr), T(req_pos)]
    casc = ra.make_cascade(*arrs, max_seg_rows=max(len(r) for _, r in segs),
                           max_seg_len=max(len(x) for x, _ in segs))
    pstart = T(start.cpu().numpy() + private)
    plen = T(np.asarray(lens) - private)
    kv2 = ra.make_kv_table(table, pstart, plen, int((np.asarray(lens) - private).max()))
    ws2 = torch.empty(ra.attn_decode_workspace(desc, B, kv2.max_len, casc), dtype=torch.uint8, device=cuda)
    cout = torch.empty_like(flat)
    clse = torch.empty_like(flat_lse)
    ra.attn_decode(desc, q, kv2, B, cout, clse, ws2, cascade=casc)
    assert ra.rc_sync(pool.err) == ra.RC_OK
    refs = _fp8_oracle_rows(pool, rows, bits(q), lens, Hq, Hkv, scale)
    check(bits(flat), refs, flat_lse.cpu().numpy(), u_p=tol.U_F16, label="flat")
    check(bits(cout), refs, clse.cpu().numpy(), u_p=tol.U_F16, label="cascade")
