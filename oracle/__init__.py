"""CPU oracle of the radix-tree KV cache and of attention: test infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product library never does, and the two
share no code: the oracle is plain C++ (pointer tree, std::map children,
std::set free list, full-scan eviction, double-precision two-pass softmax)
compiled into ``oracle/_build/liboracle.so`` by ``build()``.

Every function of the C++ side cites the passage of the pages it follows.
Parity status: every function here is pinned by tests/test_oracle_pins.py
against values the pages print (the churn counts, the cyclic sweep, the split
example), against brute force (LPM order vs all permutations, tiny
vocabularies), closed forms of attention and torch's own attention routine.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "liboracle.so")
SOURCES = ["radix_oracle.cpp", "attention_oracle.cpp"]

OK, ERR_ARG, ERR_NOMEM, ERR_STATE = 0, -1, -2, -3
FCFS, LPM = 0, 1
STAT_FIELDS = ("pool", "free", "caller", "tree_tokens", "nodes", "match_calls", "match_tokens",
               "match_hits", "match_hit_tokens", "insert_calls", "insert_new_tokens",
               "insert_dup_freed", "evicted_nodes", "evicted_tokens", "pins", "clock")


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (OpenMP on).  Returns the library path."""
    srcs = [os.path.join(HERE, s) for s in SOURCES]
    if not force and os.path.exists(LIB) and all(os.path.getmtime(LIB) >= os.path.getmtime(s) for s in srcs):
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    tmp = LIB + f".tmp{os.getpid()}"
    subprocess.check_call(["g++", "-O2", "-std=c++17", "-fopenmp", "-shared", "-fPIC", "-o", tmp] + srcs)
    os.replace(tmp, LIB)
    return LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        P, I64, I32, VP = C.POINTER, C.c_int64, C.c_int32, C.c_void_p
        L.oracle_tree_new.restype = VP
        L.oracle_tree_new.argtypes = [I64]
        L.oracle_tree_free.argtypes = [VP]
        L.oracle_match.argtypes = [VP, VP, I64, C.c_int, P(I64), VP, P(I64)]
        L.oracle_insert.argtypes = [VP, VP, VP, I64, C.c_int, P(I64), P(I64), VP]
        L.oracle_release.argtypes = [VP, I64]
        L.oracle_evict.argtypes = [VP, I64, P(I64), VP, I64, P(I64)]
        L.oracle_alloc.argtypes = [VP, I64, VP]
        L.oracle_free.argtypes = [VP, VP, I64]
        L.oracle_sched_order.argtypes = [VP, C.c_int, VP, VP, I32, VP]
        L.oracle_admit.argtypes = [VP, C.c_int, VP, VP, VP, I32, I32, VP, P(I32), VP, VP, VP, VP]
        L.oracle_commit.argtypes = [VP, C.c_int, VP, VP, VP, I32, VP, VP]
        L.oracle_dump.restype = I64
        L.oracle_dump.argtypes = [VP, C.c_char_p, I64]
        L.oracle_stats.argtypes = [VP, VP]
        L.oracle_attention.argtypes = [I64, VP, VP, VP, VP, VP, C.c_int, C.c_int, C.c_int, C.c_int,
                                       I64, I64, C.c_double, VP, VP]
        L.oracle_num_threads.restype = C.c_int
        L.oracle_set_threads.argtypes = [C.c_int]
        _lib = L
    return _lib


def _i32(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _ptr(a):
    return a.ctypes.data_as(C.c_void_p) if a is not None and a.size else None


class OracleTree:
    """Same method names and return shapes as the product binding's RadixCache."""

    def __init__(self, pool_slots: int):
        self._h = lib().oracle_tree_new(int(pool_slots))
        if not self._h:
            raise ValueError("bad pool size")

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h and _lib is not None:
            _lib.oracle_tree_free(h)

    def match(self, tokens, pin: bool):
        t = _i32(tokens)
        out = np.empty(max(len(t), 1), np.int32)
        m, node = C.c_int64(0), C.c_int64(-1)
        st = lib().oracle_match(self._h, _ptr(t), len(t), int(pin), C.byref(m), _ptr(out), C.byref(node))
        return st, m.value, out[:m.value].copy(), node.value

    def insert(self, tokens, slots, pin: bool):
        t, s = _i32(tokens), _i32(slots)
        assert len(t) == len(s)
        out = np.empty(max(len(t), 1), np.int32)
        present, node = C.c_int64(0), C.c_int64(-1)
        st = lib().oracle_insert(self._h, _ptr(t), _ptr(s), len(t), int(pin), C.byref(present),
                                 C.byref(node), _ptr(out))
        return st, present.value, node.value, out[:len(t)].copy()

    def release(self, node: int):
        return lib().oracle_release(self._h, int(node))

    def evict(self, n_tokens: int, log_cap: int = 4096):
        log = np.empty(max(log_cap, 1), np.int64)
        freed, cnt = C.c_int64(0), C.c_int64(0)
        st = lib().oracle_evict(self._h, int(n_tokens), C.byref(freed), _ptr(log), log_cap, C.byref(cnt))
        return st, freed.value, log[:min(cnt.value, log_cap)].copy()

    def alloc(self, n: int):
        out = np.empty(max(n, 1), np.int32)
        st = lib().oracle_alloc(self._h, int(n), _ptr(out))
        return st, (out[:n].copy() if st == OK else np.empty(0, np.int32))

    def free(self, slots):
        s = _i32(slots)
        return lib().oracle_free(self._h, _ptr(s), len(s))

    def sched_order(self, policy: int, prompts):
        flat = _i32(np.concatenate([np.asarray(p, np.int32) for p in prompts]) if prompts else [])
        lens = np.asarray([len(p) for p in prompts], np.int64)
        out = np.empty(max(len(prompts), 1), np.int32)
        st = lib().oracle_sched_order(self._h, int(policy), _ptr(flat), _ptr(lens), len(prompts), _ptr(out))
        return st, out[:len(prompts)].copy()

    def dump(self) -> str:
        n = lib().oracle_dump(self._h, None, 0)
        buf = C.create_string_buffer(int(n) + 1)
        lib().oracle_dump(self._h, buf, n + 1)
        return buf.value.decode()

    def stats(self) -> dict:
        v = np.zeros(16, np.int64)
        lib().oracle_stats(self._h, _ptr(v))
        return dict(zip(STAT_FIELDS, (int(x) for x in v)))


class OracleServer:
    """The oracle's own scheduling round and commits (oracle_admit,
    oracle_commit) over an OracleTree, with the method names a serving loop
    calls: admit(pending, policy, max_batch) -> (admitted, waiting),
    commit_prompts(batch), finish(batch).  Requests are any objects with
    tokens (prompt followed by the generated tokens), prompt_len, max_new; it
    sets matched, first, node and slots on the admitted ones."""

    def __init__(self, tree: OracleTree):
        self.cache = tree

    @staticmethod
    def _rows(reqs):
        lens = np.fromiter((r.prompt_len for r in reqs), np.int64, len(reqs))
        mnew = np.fromiter((r.max_new for r in reqs), np.int64, len(reqs))
        toks = _i32(np.concatenate([np.asarray(r.tokens[:r.prompt_len + r.max_new], np.int32) for r in reqs])
                    if reqs else [])
        off = np.concatenate([[0], np.cumsum(lens + mnew)]).astype(np.int64)
        return toks, lens, mnew, off

    def admit(self, pending: list, policy: int = LPM, max_batch: int | None = None):
        if not pending:
            return [], []
        n = len(pending)
        toks, lens, mnew, off = self._rows(pending)
        slots = np.zeros(max(int(off[-1]), 1), np.int32)
        order = np.zeros(n, np.int32)
        matched, first, node = np.zeros(n, np.int64), np.zeros(n, np.int64), np.zeros(n, np.int64)
        cnt = C.c_int32(0)
        st = lib().oracle_admit(self.cache._h, int(policy), _ptr(toks), _ptr(lens), _ptr(mnew), n, int(max_batch or 0),
                                _ptr(order), C.byref(cnt), _ptr(matched), _ptr(first), _ptr(node), _ptr(slots))
        if st != OK:
            raise RuntimeError(f"oracle_admit returned {st}")
        admitted = []
        for i in order[:cnt.value].tolist():
            r = pending[i]
            r.matched, r.first, r.node = int(matched[i]), int(first[i]), int(node[i])
            r.slots = slots[off[i]:off[i + 1]].copy()
            admitted.append(r)
        took = set(order[:cnt.value].tolist())
        return admitted, [r for i, r in enumerate(pending) if i not in took]

    def _commit(self, batch, mode):
        if not batch:
            return
        toks, lens, mnew, off = self._rows(batch)
        slots = _i32(np.concatenate([np.asarray(r.slots, np.int32) for r in batch]))
        node = np.fromiter((r.node for r in batch), np.int64, len(batch))
        st = lib().oracle_commit(self.cache._h, mode, _ptr(toks), _ptr(lens), _ptr(mnew), len(batch), _ptr(slots),
                                 _ptr(node))
        if st != OK:
            raise RuntimeError(f"oracle_commit returned {st}")
        for i, r in enumerate(batch):
            r.slots = slots[off[i]:off[i + 1]].copy()
            r.node = int(node[i])

    def commit_prompts(self, batch: list):
        self._commit(batch, 0)

    def finish(self, batch: list):
        self._commit(batch, 1)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


def set_threads(n: int) -> None:
    """Threads of later attention() calls (n <= 0: all the host's cores)."""
    lib().oracle_set_threads(int(n))


def attention(q, k, v, kv_off, ctx, q_heads, kv_heads, dk, dv, scale, latent=False):
    """Exact attention of many query rows, in double.

    q: uint16 bf16 bits [rows, Hq, dk]; k: [tokens, Hkv, dk]; v: [tokens, Hkv, dv]
    (ignored when ``latent``: V is the first dv columns of each K row).
    Row r sees tokens kv_off[r] .. kv_off[r]+ctx[r]-1.  Returns (out [rows,Hq,dv], lse [rows,Hq]).
    """
    q = np.ascontiguousarray(q, dtype=np.uint16)
    k = np.ascontiguousarray(k, dtype=np.uint16)
    rows = q.shape[0]
    kv_off = np.ascontiguousarray(kv_off, dtype=np.int64)
    ctx = np.ascontiguousarray(ctx, dtype=np.int64)
    assert kv_off.shape == (rows,) and ctx.shape == (rows,)
    if latent:
        vv, v_stride = k, kv_heads * dk
    else:
        vv = np.ascontiguousarray(v, dtype=np.uint16)
        v_stride = kv_heads * dv
    out = np.empty((rows, q_heads, dv), np.float64)
    lse = np.empty((rows, q_heads), np.float64)
    lib().oracle_attention(rows, _ptr(q), _ptr(k), vv.ctypes.data_as(C.c_void_p), _ptr(kv_off), _ptr(ctx),
                           q_heads, kv_heads, dk, dv, kv_heads * dk, v_stride, float(scale),
                           _ptr(out), _ptr(lse))
    return out, lse
