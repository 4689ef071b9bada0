"""Prefix-shared radix-tree KV cache with GB300 (sm_103a) attention kernels.

This module is the thin Python binding of the C-ABI library declared in
``include/radixattn.h`` (built in-tree as ``_build/libradixattn.so``).  It only
marshals arguments: every step of the path runs in the library, the host tree
in C++ and the data path in hand-written CUDA kernels.  There is no fallback:
if the library is missing, loading it raises.

Function names follow the header: ``rc_create``, ``rc_match_prefix``,
``rc_insert``, ``rc_release``, ``rc_evict``, ``rc_alloc``, ``rc_free``,
``sched_order``, ``rc_stats``, ``rc_dump``, ``kv_store``, ``attn_decode``,
``attn_extend``, ``rc_sync``.  ``RadixCache`` wraps a cache handle with the
host calls as methods.  Device calls take torch CUDA tensors (PyTorch is used
for device memory and streams only).
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

from . import _compile as _build

RC_OK, RC_ERR_ARG, RC_ERR_NOMEM, RC_ERR_STATE = 0, -1, -2, -3
RC_ERR_CUDA, RC_ERR_TIMEOUT, RC_ERR_DEVICE, RC_ERR_UNSUPPORTED = -4, -5, -6, -7
RC_ERR_SCRATCH = -8
RC_STATIC_SCRATCH_BYTES = 32 << 20
RC_FCFS, RC_LPM = 0, 1

I32, I64, VP = C.c_int32, C.c_int64, C.c_void_p
P = C.POINTER


class rc_pool_desc(C.Structure):
    _fields_ = [("k", VP), ("v", VP), ("n_slots", I64), ("kv_heads", I32), ("head_dim_k", I32),
                ("head_dim_v", I32), ("mla", I32), ("err", VP), ("kv_fp8", I32), ("k_scale", VP),
                ("v_scale", VP)]


class rc_attn_desc(C.Structure):
    _fields_ = [("pool", rc_pool_desc), ("q_heads", I32), ("sm_scale", C.c_float)]


class rc_kv_table(C.Structure):
    _fields_ = [("slots", VP), ("start", VP), ("len", VP), ("max_len", I32), ("table_len", I64)]


class rc_cascade(C.Structure):
    _fields_ = [("n_seg", I32), ("seg_slots", VP), ("seg_indptr", VP), ("seg_row_indptr", VP),
                ("seg_rows", VP), ("req_seg_indptr", VP), ("req_seg_pos", VP), ("max_seg_len", I32), ("max_seg_rows", I32),
                ("total_seg_rows", I32), ("host_seg_indptr", VP), ("host_seg_row_indptr", VP)]


class rc_decode_step(C.Structure):
    _fields_ = [("q", VP), ("k_new", VP), ("v_new", VP), ("store_slots", VP), ("out", VP), ("lse", VP),
                ("len", VP), ("max_len", I32), ("ev_begin", VP), ("ev_end", VP)]


class rc_request(C.Structure):
    _fields_ = [("tokens", VP), ("prompt_len", I64), ("max_new", I64), ("slots", VP), ("matched", I64),
                ("first", I64), ("node", I64), ("admitted", I32)]


RC_COMMIT_PREFILL, RC_COMMIT_FINISH = 0, 1


class rc_stats_t(C.Structure):
    _fields_ = [(n, I64) for n in (
        "pool_slots", "free_slots", "caller_slots", "tree_tokens", "nodes", "match_calls", "match_tokens",
        "match_hits", "match_hit_tokens", "insert_calls", "insert_new_tokens", "insert_dup_freed",
        "evicted_nodes", "evicted_tokens", "pins", "clock")]


# header declarations: name -> (restype, argtypes)
SIGNATURES = {
    "rc_create": (I32, [I64, P(VP)]),
    "rc_destroy": (None, [VP]),
    "rc_match_prefix": (I32, [VP, VP, I64, C.c_int, P(I64), VP, P(I64)]),
    "rc_insert": (I32, [VP, VP, VP, I64, C.c_int, P(I64), P(I64), VP]),
    "rc_release": (I32, [VP, I64]),
    "rc_evict": (I32, [VP, I64, P(I64), VP, I64, P(I64)]),
    "rc_alloc": (I32, [VP, I64, VP]),
    "rc_free": (I32, [VP, VP, I64]),
    "sched_order": (I32, [VP, C.c_int, VP, VP, I32, VP]),
    "rc_stats": (I32, [VP, P(rc_stats_t)]),
    "rc_admit": (I32, [VP, C.c_int, VP, I32, I32, VP, P(I32)]),
    "rc_commit": (I32, [VP, VP, VP, I32, C.c_int]),
    "rc_cascade_plan": (I32, [VP, VP, I32, VP, I64, VP, VP, VP, VP, VP, I64, VP, I32, P(I32), P(I64), P(I32),
                              P(I32), P(I32)]),
    "rc_dump": (I32, [VP, C.c_char_p, I64, P(I64)]),
    "kv_store": (I32, [P(rc_pool_desc), VP, VP, VP, I32, VP, VP, VP]),
    "attn_decode_workspace": (I32, [P(rc_attn_desc), I32, I32, P(rc_cascade), P(C.c_size_t)]),
    "attn_decode": (I32, [P(rc_attn_desc), VP, P(rc_kv_table), I32, P(rc_cascade), VP, VP, VP, C.c_size_t, VP]),
    "attn_decode_append": (I32, [P(rc_attn_desc), VP, VP, VP, P(rc_kv_table), I32, P(rc_cascade), VP, VP, VP,
                                 C.c_size_t, VP]),
    "attn_decode_steps": (I32, [P(rc_attn_desc), P(rc_kv_table), I32, P(rc_cascade), P(rc_decode_step), I32, VP,
                                C.c_size_t, VP, P(I32)]),
    "attn_decode_static": (I32, [P(rc_attn_desc), VP, P(rc_kv_table), I32, P(rc_cascade), VP, VP, VP]),
    "attn_extend_workspace": (I32, [P(rc_attn_desc), I32, I32, I32, P(C.c_size_t)]),
    "attn_extend": (I32, [P(rc_attn_desc), VP, VP, P(rc_kv_table), I32, I32, VP, VP, VP, C.c_size_t, VP]),
    "rc_sync": (I32, [VP, VP]),
    "rc_probe_wait_timeout": (I32, [VP, VP]),
    "rc_strerror": (C.c_char_p, [I32]),
    "rc_image_key": (I32, [VP, I64, I32, VP]),
    "bc_create": (I32, [I64, I32, P(VP)]),
    "bc_destroy": (None, [VP]),
    "bc_match_prefix": (I32, [VP, VP, I64, C.c_int, P(I64), VP, P(I64)]),
    "bc_insert": (I32, [VP, VP, VP, I64, C.c_int, P(I64), P(I64), VP]),
    "bc_release": (I32, [VP, I64]),
    "bc_evict": (I32, [VP, I64, P(I64), VP, I64, P(I64)]),
    "bc_alloc": (I32, [VP, I64, VP]),
    "bc_free": (I32, [VP, VP, I64]),
    "bc_sched_order": (I32, [VP, C.c_int, VP, VP, I32, VP]),
    "bc_stats": (I32, [VP, P(rc_stats_t)]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Load the C-ABI library; raises if it has not been built."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; "
                               "g.build()' or python -m radixattention_prefix_shared_tree_gb300._compile)")
        L = C.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def rc_strerror(status: int) -> str:
    return lib().rc_strerror(int(status)).decode()


class RCError(RuntimeError):
    def __init__(self, call, status):
        super().__init__(f"{call}: {rc_strerror(status)} ({status})")
        self.status = status


def _check(call, st):
    if st != RC_OK:
        raise RCError(call, st)


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _np_ptr(a):
    return a.ctypes.data_as(VP) if a is not None and a.size else None


# ------------------------------------------------------------------ host calls
def rc_create(pool_slots: int):
    h = VP()
    st = lib().rc_create(int(pool_slots), C.byref(h))
    _check("rc_create", st)
    return h


def rc_destroy(handle):
    lib().rc_destroy(handle)


def rc_match_prefix(handle, tokens, pin: bool, _fn: str = "rc_match_prefix"):
    t = _i32(tokens)
    out = np.empty(max(len(t), 1), np.int32)
    m, node = I64(0), I64(-1)
    st = getattr(lib(), _fn)(handle, _np_ptr(t), len(t), int(pin), C.byref(m), out.ctypes.data_as(VP),
                             C.byref(node))
    return st, m.value, out[:m.value].copy(), node.value


def rc_insert(handle, tokens, slots, pin: bool, _fn: str = "rc_insert"):
    t, s = _i32(tokens), _i32(slots)
    if len(t) != len(s):
        raise ValueError("tokens and slots differ in length")
    out = np.empty(max(len(t), 1), np.int32)
    present, node = I64(0), I64(-1)
    st = getattr(lib(), _fn)(handle, _np_ptr(t), _np_ptr(s), len(t), int(pin), C.byref(present), C.byref(node),
                             out.ctypes.data_as(VP))
    return st, present.value, node.value, out[:len(t)].copy()


def rc_release(handle, node: int, _fn: str = "rc_release"):
    return getattr(lib(), _fn)(handle, int(node))


def rc_evict(handle, n_tokens: int, log_cap: int = 4096, _fn: str = "rc_evict"):
    log = np.empty(max(log_cap, 1), np.int64)
    freed, cnt = I64(0), I64(0)
    st = getattr(lib(), _fn)(handle, int(n_tokens), C.byref(freed), log.ctypes.data_as(VP), log_cap, C.byref(cnt))
    return st, freed.value, log[:min(cnt.value, log_cap)].copy()


def rc_alloc(handle, n: int, _fn: str = "rc_alloc"):
    out = np.empty(max(n, 1), np.int32)
    st = getattr(lib(), _fn)(handle, int(n), out.ctypes.data_as(VP))
    return st, (out[:n].copy() if st == RC_OK else np.empty(0, np.int32))


def rc_free(handle, slots, _fn: str = "rc_free"):
    s = _i32(slots)
    return getattr(lib(), _fn)(handle, _np_ptr(s), len(s))


def sched_order(handle, policy: int, prompts, _fn: str = "sched_order"):
    arrs = [_i32(p) for p in prompts]
    ptrs = (VP * max(len(arrs), 1))(*[a.ctypes.data if a.size else None for a in arrs])
    lens = np.asarray([len(a) for a in arrs], np.int64)
    out = np.empty(max(len(arrs), 1), np.int32)
    st = getattr(lib(), _fn)(handle, int(policy), ptrs, _np_ptr(lens), len(arrs), out.ctypes.data_as(VP))
    return st, out[:len(arrs)].copy()


def rc_stats(handle, _fn: str = "rc_stats") -> dict:
    s = rc_stats_t()
    _check(_fn, getattr(lib(), _fn)(handle, C.byref(s)))
    return {n: int(getattr(s, n)) for n, _ in rc_stats_t._fields_}


def rc_image_key(data, n_tokens: int):
    """Key run of an image (bytes-like or numpy array) for the tree."""
    buf = np.frombuffer(bytes(data), np.uint8) if not isinstance(data, np.ndarray) else \
        np.ascontiguousarray(data).view(np.uint8).reshape(-1)
    out = np.empty(max(int(n_tokens), 1), np.int32)
    _check("rc_image_key", lib().rc_image_key(_np_ptr(buf), buf.size, int(n_tokens), out.ctypes.data_as(VP)))
    return out[:int(n_tokens)].copy()


def rc_dump(handle) -> str:
    need = I64(0)
    _check("rc_dump", lib().rc_dump(handle, None, 0, C.byref(need)))
    buf = C.create_string_buffer(need.value + 1)
    _check("rc_dump", lib().rc_dump(handle, buf, need.value + 1, C.byref(need)))
    return buf.value.decode()


def _req_ptr(reqs):
    """Address of an rc_request array: a ctypes array, or a numpy structured
    array with the same record layout."""
    return reqs.ctypes.data if isinstance(reqs, np.ndarray) else C.cast(reqs, VP)


def rc_admit(handle, policy: int, reqs, n: int, max_batch: int, out_order):
    """reqs: array of rc_request (see _req_ptr); out_order: int32 numpy array of n."""
    cnt = I32(0)
    st = lib().rc_admit(handle, int(policy), _req_ptr(reqs), int(n), int(max_batch), _np_ptr(out_order),
                        C.byref(cnt))
    return st, cnt.value


def rc_cascade_plan(handle, nodes):
    """Cascade segments of the requests pinned at `nodes` (see the header).
    Returns a dict of numpy arrays and bounds."""
    nodes = np.ascontiguousarray(nodes, dtype=np.int64)
    n = len(nodes)
    cap_slots, cap_rows, cap_seg = 1 << 16, 1 << 12, 1 << 10
    while True:
        seg_slots = np.empty(cap_slots, np.int32)
        seg_indptr = np.empty(cap_seg + 1, np.int32)
        seg_row_indptr = np.empty(cap_seg + 1, np.int32)
        seg_rows = np.empty(cap_rows, np.int32)
        req_seg_pos = np.empty(cap_rows, np.int32)
        req_seg_indptr = np.empty(n + 1, np.int32)
        private = np.empty(max(n, 1), np.int64)
        ns, nsl, tot, mlen, mrows = I32(0), I64(0), I32(0), I32(0), I32(0)
        st = lib().rc_cascade_plan(handle, _np_ptr(nodes), n, _np_ptr(seg_slots), cap_slots, _np_ptr(seg_indptr),
                                   _np_ptr(seg_row_indptr), _np_ptr(seg_rows), _np_ptr(req_seg_indptr),
                                   _np_ptr(req_seg_pos), cap_rows, _np_ptr(private), cap_seg, C.byref(ns),
                                   C.byref(nsl), C.byref(tot), C.byref(mlen), C.byref(mrows))
        if st == RC_ERR_NOMEM:
            cap_slots, cap_rows, cap_seg = cap_slots * 8, cap_rows * 8, cap_seg * 8
            continue
        _check("rc_cascade_plan", st)
        k = ns.value
        return dict(n_seg=k, seg_slots=seg_slots[:nsl.value], seg_indptr=seg_indptr[:k + 1],
                    seg_row_indptr=seg_row_indptr[:k + 1], seg_rows=seg_rows[:tot.value],
                    req_seg_indptr=req_seg_indptr, req_seg_pos=req_seg_pos[:tot.value], private=private[:n],
                    max_seg_len=mlen.value, max_seg_rows=mrows.value)


def rc_commit(handle, reqs, idx, mode: int):
    idx = _i32(idx)
    return lib().rc_commit(handle, _req_ptr(reqs), _np_ptr(idx), len(idx), int(mode))


_STAT_RENAME = {"pool_slots": "pool", "free_slots": "free", "caller_slots": "caller"}


class RadixCache:
    """A cache handle with the host calls as methods (same shapes as the oracle's tree)."""

    def __init__(self, pool_slots: int):
        self._h = rc_create(pool_slots)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.rc_destroy(h)

    @property
    def handle(self):
        return self._h

    def match(self, tokens, pin: bool):
        return rc_match_prefix(self._h, tokens, pin)

    def insert(self, tokens, slots, pin: bool):
        return rc_insert(self._h, tokens, slots, pin)

    def release(self, node: int):
        return rc_release(self._h, node)

    def evict(self, n_tokens: int, log_cap: int = 4096):
        return rc_evict(self._h, n_tokens, log_cap)

    def alloc(self, n: int):
        return rc_alloc(self._h, n)

    def free(self, slots):
        return rc_free(self._h, slots)

    def sched_order(self, policy: int, prompts):
        return sched_order(self._h, policy, prompts)

    def dump(self) -> str:
        return rc_dump(self._h)

    # batched calls used by the scheduler's fast path
    def admit_batch(self, policy, reqs, n, max_batch, out_order):
        return rc_admit(self._h, policy, reqs, n, max_batch, out_order)

    def commit_batch(self, reqs, idx, mode):
        return rc_commit(self._h, reqs, idx, mode)

    def cascade_plan(self, nodes):
        return rc_cascade_plan(self._h, nodes)

    def stats(self) -> dict:
        return {_STAT_RENAME.get(k, k): v for k, v in rc_stats(self._h).items()}


class BlockCache:
    """The block-granular comparator (bc_* calls) with RadixCache's method
    shapes; ``uncached_tail(n)`` is how many of n inserted tokens stay with the
    caller (the partial last block)."""

    def __init__(self, pool_slots: int, block_tokens: int = 16):
        h = VP()
        _check("bc_create", lib().bc_create(int(pool_slots), int(block_tokens), C.byref(h)))
        self._h = h
        self.block_tokens = int(block_tokens)

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.bc_destroy(h)

    @property
    def handle(self):
        return self._h

    def match(self, tokens, pin: bool):
        return rc_match_prefix(self._h, tokens, pin, _fn="bc_match_prefix")

    def insert(self, tokens, slots, pin: bool):
        return rc_insert(self._h, tokens, slots, pin, _fn="bc_insert")

    def release(self, node: int):
        return rc_release(self._h, node, _fn="bc_release")

    def evict(self, n_tokens: int, log_cap: int = 4096):
        return rc_evict(self._h, n_tokens, log_cap, _fn="bc_evict")

    def alloc(self, n: int):
        return rc_alloc(self._h, n, _fn="bc_alloc")

    def free(self, slots):
        return rc_free(self._h, slots, _fn="bc_free")

    def sched_order(self, policy: int, prompts):
        return sched_order(self._h, policy, prompts, _fn="bc_sched_order")

    def uncached_tail(self, n: int) -> int:
        return int(n) % self.block_tokens

    def stats(self) -> dict:
        return {_STAT_RENAME.get(k, k): v for k, v in rc_stats(self._h, _fn="bc_stats").items()}


# ---------------------------------------------------------------- device calls
def _tp(t):
    """Device pointer of a torch tensor (None -> NULL).  The kernels read and
    write dense row-major arrays, so a strided view is refused rather than
    misread."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError(f"expected a contiguous tensor, got shape {tuple(t.shape)} strides {t.stride()}")
    return C.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return C.c_void_p(s.cuda_stream)


def make_pool_desc(k, v, err=None, mla: bool = False, head_dim_v: int | None = None, k_scale=None,
                   v_scale=None) -> rc_pool_desc:
    """Descriptor of a pool held in torch tensors: k [n_slots, Hkv, dk] (or [n_slots, dk] latent).
    With k_scale / v_scale (fp32 [n_slots, Hkv]) the pool is FP8: k, v hold E4M3 codes (uint8).
    The kernels index the pool as dense row-major arrays, so every tensor must be contiguous."""
    for name, t in (("k", k), ("v", v), ("k_scale", k_scale), ("v_scale", v_scale)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"make_pool_desc: {name} must be contiguous (dense row-major [n_slots, ...])")
    d = rc_pool_desc()
    d.k = k.data_ptr()
    d.v = v.data_ptr() if v is not None else None
    d.n_slots = k.shape[0]
    if mla:
        d.kv_heads, d.head_dim_k = 1, k.shape[-1]
        d.head_dim_v = int(head_dim_v)
    else:
        d.kv_heads, d.head_dim_k = k.shape[1], k.shape[2]
        d.head_dim_v = v.shape[2]
    d.mla = int(mla)
    d.err = err.data_ptr() if err is not None else None
    if k_scale is not None:
        d.kv_fp8 = 1
        d.k_scale, d.v_scale = k_scale.data_ptr(), v_scale.data_ptr()
    d._keep = (k, v, err, k_scale, v_scale)   # raw pointers inside: keep the tensors alive with it
    return d


def make_attn_desc(pool: rc_pool_desc, q_heads: int, sm_scale: float) -> rc_attn_desc:
    a = rc_attn_desc()
    a.pool = pool
    a.q_heads = int(q_heads)
    a.sm_scale = float(sm_scale)
    a._keep = getattr(pool, "_keep", None)
    return a


def make_kv_table(slots, start, length, max_len: int, table_len: int | None = None) -> rc_kv_table:
    t = rc_kv_table()
    t.slots, t.start, t.len = slots.data_ptr(), start.data_ptr(), length.data_ptr()
    t.max_len = int(max_len)
    t.table_len = int(slots.numel() if table_len is None else table_len)
    t._keep = (slots, start, length)   # raw pointers inside: keep the tensors alive with it
    return t


def make_cascade(seg_slots, seg_indptr, seg_row_indptr, seg_rows, req_seg_indptr, req_seg_pos,
                 max_seg_rows: int, max_seg_len: int, host_seg_indptr=None, host_seg_row_indptr=None) -> rc_cascade:
    """Device arrays as tensors; host_seg_indptr / host_seg_row_indptr: None,
    or numpy copies of seg_indptr / seg_row_indptr (the grid then covers the
    non-empty segment chunks only)."""
    c = rc_cascade()
    host = ()
    if host_seg_indptr is not None and host_seg_row_indptr is not None:
        host = (np.ascontiguousarray(host_seg_indptr, np.int32), np.ascontiguousarray(host_seg_row_indptr, np.int32))
        c.host_seg_indptr = host[0].ctypes.data
        c.host_seg_row_indptr = host[1].ctypes.data
    c.n_seg = seg_indptr.numel() - 1
    c.seg_slots = seg_slots.data_ptr() if seg_slots.numel() else None
    c.seg_indptr, c.seg_row_indptr = seg_indptr.data_ptr(), seg_row_indptr.data_ptr()
    c.seg_rows = seg_rows.data_ptr() if seg_rows.numel() else None
    c.req_seg_indptr = req_seg_indptr.data_ptr()
    c.req_seg_pos = req_seg_pos.data_ptr() if req_seg_pos.numel() else None
    c.max_seg_rows = int(max_seg_rows)
    c.max_seg_len = int(max_seg_len)
    c.total_seg_rows = int(seg_rows.numel())
    c._keep = (seg_slots, seg_indptr, seg_row_indptr, seg_rows, req_seg_indptr, req_seg_pos) + host
    return c


def kv_store(pool: rc_pool_desc, slots, k_new, v_new, table=None, table_pos=None, stream=None):
    st = lib().kv_store(C.byref(pool), _tp(slots), _tp(k_new), _tp(v_new), int(slots.numel()), _tp(table),
                        _tp(table_pos), _stream(stream))
    _check("kv_store", st)


def attn_decode_workspace(desc: rc_attn_desc, batch: int, max_len: int, cascade: rc_cascade | None = None) -> int:
    n = C.c_size_t(0)
    st = lib().attn_decode_workspace(C.byref(desc), int(batch), int(max_len),
                                     C.byref(cascade) if cascade is not None else None, C.byref(n))
    _check("attn_decode_workspace", st)
    return int(n.value)


def attn_decode(desc: rc_attn_desc, q, kv: rc_kv_table, batch: int, out, lse=None, ws=None,
                cascade: rc_cascade | None = None, stream=None):
    st = lib().attn_decode(C.byref(desc), _tp(q), C.byref(kv), int(batch),
                           C.byref(cascade) if cascade is not None else None, _tp(out), _tp(lse), _tp(ws),
                           int(ws.numel() * ws.element_size()) if ws is not None else 0, _stream(stream))
    _check("attn_decode", st)


def attn_decode_append(desc: rc_attn_desc, q, k_new, v_new, kv: rc_kv_table, batch: int, out, lse=None, ws=None,
                       cascade: rc_cascade | None = None, stream=None):
    """attn_decode that also stores each row's last key from k_new/v_new
    ([batch][kv_heads][head_dim] bf16) into its pool slot (see the header)."""
    st = lib().attn_decode_append(C.byref(desc), _tp(q), _tp(k_new), _tp(v_new), C.byref(kv), int(batch),
                                  C.byref(cascade) if cascade is not None else None, _tp(out), _tp(lse), _tp(ws),
                                  int(ws.numel() * ws.element_size()) if ws is not None else 0, _stream(stream))
    _check("attn_decode_append", st)


def attn_decode_steps(desc: rc_attn_desc, kv: rc_kv_table, batch: int, steps, ws=None,
                      cascade: rc_cascade | None = None, stream=None):
    """Several decode steps of one batch in one call.  steps: a list of dicts
    with q, out and len (tensors), max_len (int), and optionally k_new/v_new,
    store_slots, lse (tensors): each step as attn_decode_append (k_new given),
    kv_store + attn_decode (store_slots given) or attn_decode (see the header)."""
    arr = (rc_decode_step * max(len(steps), 1))()
    for i, s in enumerate(steps):
        a = arr[i]
        a.q, a.out, a.len, a.max_len = _tp(s["q"]), _tp(s["out"]), _tp(s["len"]), int(s["max_len"])
        a.k_new, a.v_new = _tp(s.get("k_new")), _tp(s.get("v_new"))
        a.store_slots, a.lse = _tp(s.get("store_slots")), _tp(s.get("lse"))
    done = I32(0)
    st = lib().attn_decode_steps(C.byref(desc), C.byref(kv), int(batch),
                                 C.byref(cascade) if cascade is not None else None, arr, len(steps), _tp(ws),
                                 int(ws.numel() * ws.element_size()) if ws is not None else 0, _stream(stream),
                                 C.byref(done))
    _check("attn_decode_steps", st)


def attn_decode_static(desc: rc_attn_desc, q, kv: rc_kv_table, batch: int, out, lse=None,
                       cascade: rc_cascade | None = None, stream=None) -> int:
    """attn_decode with the library's fixed scratch area (no workspace, no
    allocation).  Returns the status instead of raising, so callers can see
    RC_ERR_SCRATCH."""
    return lib().attn_decode_static(C.byref(desc), _tp(q), C.byref(kv), int(batch),
                                    C.byref(cascade) if cascade is not None else None, _tp(out), _tp(lse),
                                    _stream(stream))


def attn_extend_workspace(desc: rc_attn_desc, batch: int, max_q: int, max_len: int) -> int:
    n = C.c_size_t(0)
    _check("attn_extend_workspace", lib().attn_extend_workspace(C.byref(desc), int(batch), int(max_q),
                                                                 int(max_len), C.byref(n)))
    return int(n.value)


def attn_extend(desc: rc_attn_desc, q, qo_indptr, kv: rc_kv_table, batch: int, max_q: int, out, lse=None,
                ws=None, stream=None):
    st = lib().attn_extend(C.byref(desc), _tp(q), _tp(qo_indptr), C.byref(kv), int(batch), int(max_q), _tp(out),
                           _tp(lse), _tp(ws), int(ws.numel() * ws.element_size()) if ws is not None else 0,
                           _stream(stream))
    _check("attn_extend", st)


def rc_sync(err=None, stream=None) -> int:
    return lib().rc_sync(_stream(stream), _tp(err))


def rc_probe_wait_timeout(err, stream=None) -> int:
    """Launch the bounded-wait self-test (see the header); rc_sync(err) then
    returns RC_ERR_TIMEOUT."""
    return lib().rc_probe_wait_timeout(_tp(err), _stream(stream))
