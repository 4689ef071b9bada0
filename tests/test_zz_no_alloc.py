"""attn_decode_static: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc or hand the library a workspace (a serving
loop whose device memory is all carved up at start-up, a host framework whose
plugin interface passes only input and output pointers).  For them the
library keeps the split partials in a fixed device array of its own.  This
file checks, through the C ABI, that two calls in a row give the same result
as attn_decode with a caller workspace, and that a batch needing more scratch
than the fixed area is refused.  It runs last (file name) and also passes on
its own in a fresh process.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import radixattention_prefix_shared_tree_gb300 as ra
from radixattention_prefix_shared_tree_gb300.driver import plan_cascade
from synth import hashgen as hg

pytestmark = pytest.mark.gpu

def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _case(dev, seed, Hq, Hkv, D, lens, n_slots=12000):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(n_slots, Hkv, D, generator=g).to(torch.bfloat16).to(dev)
    v = torch.randn(n_slots, Hkv, D, generator=g).to(torch.bfloat16).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    rng = np.random.default_rng(seed)
    shared = rng.choice(n_slots, size=600, replace=False).astype(np.int32)
    rest = np.setdiff1d(np.arange(n_slots, dtype=np.int32), shared)
    rng.shuffle(rest)
    rows, off = [], 0
    for L in lens:
        rows.append(np.concatenate([shared, rest[off:off + L]]).astype(np.int32))
        off += L
    B = len(rows)
    full = [len(r) for r in rows]
    starts = np.concatenate([[0], np.cumsum(full)[:-1]]).astype(np.int32)
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    state = dict(k=k, v=v, err=err, table=T(np.concatenate(rows)), start=T(starts), len=T(full))
    state["pool"] = ra.make_pool_desc(k, v, err)
    state["desc"] = ra.make_attn_desc(state["pool"], Hq, 1.0 / np.sqrt(D))
    state["kv"] = ra.make_kv_table(state["table"], state["start"], state["len"], max(full))
    state["q"] = torch.randn(B, Hq, D, generator=g).to(torch.bfloat16).to(dev)
    # cascade over the shared part (the last position of every row stays private)
    segs, private = plan_cascade([r[:-1] for r in rows])
    seg_rows = np.concatenate([np.asarray(r, np.int32) for _, r in segs])
    pos_of = [[p for p, b in enumerate(seg_rows) if b == bb] for bb in range(B)]
    arrs = [T(np.concatenate([s for s, _ in segs])), T(np.concatenate([[0], np.cumsum([len(s) for s, _ in segs])])),
            T(np.concatenate([[0], np.cumsum([len(r) for _, r in segs])])), T(seg_rows),
            T(np.concatenate([[0], np.cumsum([len(x) for x in pos_of])])), T(np.concatenate(pos_of))]
    state["casc_arrays"] = arrs
    state["casc"] = ra.make_cascade(*arrs, max_seg_rows=max(len(r) for _, r in segs),
                           max_seg_len=max(len(x) for x, _ in segs))
    state["pstart"], state["plen"] = T(starts + private), T(np.asarray(full) - private)
    state["kv_tail"] = ra.make_kv_table(state["table"], state["pstart"], state["plen"],
                                        int((np.asarray(full) - private).max()))
    state["B"] = B
    return state


def _with_workspace(st, cascade):
    kv, casc = (st["kv_tail"], st["casc"]) if cascade else (st["kv"], None)
    n = ra.attn_decode_workspace(st["desc"], st["B"], kv.max_len, casc)
    ws = torch.empty(n, dtype=torch.uint8, device=st["q"].device)
    out = torch.empty(st["B"], st["q"].shape[1], st["q"].shape[2], dtype=torch.bfloat16, device=ws.device)
    lse = torch.empty(st["B"], st["q"].shape[1], dtype=torch.float32, device=ws.device)
    ra.attn_decode(st["desc"], st["q"], kv, st["B"], out, lse, ws, cascade=casc)
    return out, lse


def _static(st, cascade):
    kv, casc = (st["kv_tail"], st["casc"]) if cascade else (st["kv"], None)
    out = torch.empty(st["B"], st["q"].shape[1], st["q"].shape[2], dtype=torch.bfloat16, device=st["q"].device)
    lse = torch.empty(st["B"], st["q"].shape[1], dtype=torch.float32, device=out.device)
    status = ra.attn_decode_static(st["desc"], st["q"], kv, st["B"], out, lse, cascade=casc)
    assert status == ra.RC_OK, ra.rc_strerror(status)
    return out, lse


def _same(a, b):
    """The fixed-scratch call runs the same kernels on the same plan and
    partial layout as the caller-workspace call: outputs and LSE bit for bit."""
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16))
    assert torch.equal(a[1].view(torch.int32), b[1].view(torch.int32))


@pytest.mark.parametrize("cascade", [False, True])
def test_static_scratch_matches_workspace_twice(cascade):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    a = _case(dev, 1, 32, 8, 128, [1, 40, 300, 1500, 77, 5])
    b = _case(dev, 2, 64, 8, 128, [900, 3, 64, 65])
    for st in (a, b):          # two calls in a row, different batches, shared scratch reused
        ref = _with_workspace(st, cascade)
        got = _static(st, cascade)
        torch.cuda.synchronize()
        _same(got, ref)
        assert ra.rc_sync(st["err"]) == ra.RC_OK
    again = _static(a, cascade)   # and back to the first batch after the second overwrote the scratch
    _same(again, _with_workspace(a, cascade))


def test_static_scratch_refuses_oversized_batch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    st = _case(dev, 3, 32, 8, 128, [10, 10])
    # a batch whose partials exceed the fixed area (4096 rows reading one
    # shared segment): refused before any launch
    big_b = 4096
    kv = ra.make_kv_table(st["table"], st["start"], st["len"], 64)
    casc = ra.rc_cascade()
    casc.n_seg, casc.max_seg_len, casc.max_seg_rows, casc.total_seg_rows = 1, 1000, big_b, big_b
    for name, t in zip(("seg_slots", "seg_indptr", "seg_row_indptr", "seg_rows", "req_seg_indptr", "req_seg_pos"),
                       st["casc_arrays"]):
        setattr(casc, name, t.data_ptr())
    need = ra.attn_decode_workspace(st["desc"], big_b, 64, casc)
    assert need > ra.RC_STATIC_SCRATCH_BYTES
    out = torch.empty(1, dtype=torch.bfloat16, device=dev)
    assert ra.attn_decode_static(st["desc"], st["q"], kv, big_b, out, cascade=casc) == ra.RC_ERR_SCRATCH
    assert "scratch" in ra.rc_strerror(ra.RC_ERR_SCRATCH)


def _latent_case(dev, seed, lens, n_slots=9000):
    """One 576-wide latent KV head, 128 query heads (the latent kernels)."""
    g = torch.Generator().manual_seed(seed)
    pool = torch.randn(n_slots, 576, generator=g).to(torch.bfloat16).to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    pd = ra.make_pool_desc(pool, None, err, mla=True, head_dim_v=512)
    rng = np.random.default_rng(seed)
    rows = [rng.choice(n_slots, size=L, replace=False).astype(np.int32) for L in lens]
    T = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)
    st = dict(pool_t=pool, err=err, pool=pd, table=T(np.concatenate(rows)),
              start=T(np.concatenate([[0], np.cumsum(lens)[:-1]])), len=T(lens), B=len(lens))
    st["desc"] = ra.make_attn_desc(pd, 128, 1.0 / np.sqrt(576))
    st["kv"] = ra.make_kv_table(st["table"], st["start"], st["len"], max(lens))
    st["q"] = torch.randn(len(lens), 128, 576, generator=g).to(torch.bfloat16).to(dev)
    return st


def _latent_pair(st):
    B, dev = st["B"], st["q"].device
    n = ra.attn_decode_workspace(st["desc"], B, st["kv"].max_len)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    outs = []
    for static in (False, True):
        out = torch.empty(B, 128, 512, dtype=torch.bfloat16, device=dev)
        lse = torch.empty(B, 128, dtype=torch.float32, device=dev)
        if static:
            status = ra.attn_decode_static(st["desc"], st["q"], st["kv"], B, out, lse)
            assert status == ra.RC_OK, ra.rc_strerror(status)
        else:
            ra.attn_decode(st["desc"], st["q"], st["kv"], B, out, lse, ws)
        outs.append((out, lse))
    assert ra.rc_sync(st["err"]) == ra.RC_OK
    return outs


def test_static_scratch_latent_and_fp8_pool_twice():
    """The latent layout (its own kernels and partial layout) and an E4M3
    pool through the fixed scratch, two batches in a row each, bit for bit
    against the caller-workspace call."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    for lens in ([700, 33, 2500], [1, 4100]):   # split chunks and a merge in both
        got, ref = _latent_pair(_latent_case(dev, len(lens), lens))
        _same(got, ref)
    # E4M3 pool: codes and scales written by kv_store from a bf16 case
    for seed, lens in ((4, [1, 40, 300, 1500, 77, 5]), (5, [900, 3, 64, 65])):
        st = _case(dev, seed, 32, 8, 128, lens)
        n_slots = st["k"].shape[0]
        k8 = torch.zeros(n_slots, 8, 128, dtype=torch.uint8, device=dev)
        v8 = torch.zeros_like(k8)
        ks = torch.zeros(n_slots, 8, dtype=torch.float32, device=dev)
        vs = torch.zeros_like(ks)
        pool8 = ra.make_pool_desc(k8, v8, st["err"], k_scale=ks, v_scale=vs)
        slots = torch.arange(n_slots, dtype=torch.int32, device=dev)
        ra.kv_store(pool8, slots, st["k"], st["v"])
        st["desc"] = ra.make_attn_desc(pool8, 32, 1.0 / np.sqrt(128))
        st["_keep"] = (k8, v8, ks, vs, pool8)
        for cascade in (False, True):
            _same(_static(st, cascade), _with_workspace(st, cascade))
        assert ra.rc_sync(st["err"]) == ra.RC_OK
