"""Request driver over the C-ABI: admission, prefill, decode and finish.

Host side (``Scheduler``): works with any object that has the cache calls of
``RadixCache`` (the oracle's tree has the same shape, which is how the tests
replay one trace through both and compare every result).  The rules it
applies around the cache calls:

* admission runs in ``sched_order`` order and stops at the first request that
  does not fit, after evicting least-recently-used leaves for it
  (inference-notes note 49, sections 4 and 5);
* a request that will decode and whose whole prompt is cached recomputes its
  last prompt token, so that one new token carries the query; that token's
  fresh slot is a duplicate that ``rc_insert`` frees;
* slots for every position the request will ever compute (uncached prompt
  tail + max_new decode tokens) are taken at admission, so the slot row of a
  request is complete before its first kernel runs;
* after prefill the prompt is inserted and stays pinned (concurrent requests
  can share it); at finish prompt + generated tokens are inserted (note 49,
  section 2: a finished request's path, outputs included, stays) and the pin
  is dropped.

Device side (``DeviceEngine``): the KV pool, the slot tables and the kernel
launches; PyTorch only provides device memory and the stream.
"""
from __future__ import annotations

import ctypes as C
import sys
import threading
import time
from dataclasses import dataclass, field

import numpy as np

from . import (RC_COMMIT_FINISH, RC_COMMIT_PREFILL, RC_ERR_NOMEM, RC_FCFS, RC_LPM, RC_OK, RCError, attn_decode,
               attn_decode_workspace, attn_extend, kv_store, lib, make_attn_desc, make_cascade, make_kv_table,
               make_pool_desc, rc_decode_step, rc_request)


@dataclass
class Request:
    rid: int
    tokens: np.ndarray          # prompt followed by the tokens it will generate (int32)
    prompt_len: int
    max_new: int
    node: int = -1              # pinned node
    matched: int = 0            # cached prefix length found at admission
    first: int = 0              # first position computed by prefill
    slots: np.ndarray = field(default_factory=lambda: np.zeros(0, np.int32))  # one per position

    @property
    def prompt(self) -> np.ndarray:
        return self.tokens[:self.prompt_len]

    @property
    def n_new(self) -> int:
        return self.prompt_len - self.first

    def tokens_addr(self) -> int:
        """Address of `tokens` for the native calls (made int32 and
        C-contiguous first if it is not), kept while the array stays the same."""
        c = self.__dict__.get("_addr")
        t = self.tokens
        if c is None or c[0] is not t:
            if t.dtype != np.int32 or not t.flags.c_contiguous:
                t = self.tokens = np.ascontiguousarray(t, np.int32)
            c = self._addr = (t, t.ctypes.data)
        return c[1]


def _tokens_addr(r) -> int:
    """Request.tokens_addr for any object with a `tokens` array."""
    f = getattr(r, "tokens_addr", None)
    if f is not None:
        return f()
    if r.tokens.dtype != np.int32 or not r.tokens.flags.c_contiguous:
        r.tokens = np.ascontiguousarray(r.tokens, np.int32)
    return r.tokens.ctypes.data


class SchedulerError(RuntimeError):
    pass


class AdmitRound:
    """One native admission round: the rc_request records (numpy, the
    library's layout) and the flat array that holds every request's slot row
    (row i at flat[off[i]:off[i+1]], written by rc_admit and rc_commit)."""

    __slots__ = ("req", "flat", "off")

    def __init__(self, req, flat, off):
        self.req, self.flat, self.off = req, flat, off


# record layout of rc_request (checked against the ctypes structure below)
_REQ_DTYPE = np.dtype([("tokens", "u8"), ("prompt_len", "i8"), ("max_new", "i8"), ("slots", "u8"),
                       ("matched", "i8"), ("first", "i8"), ("node", "i8"), ("admitted", "i4"), ("_pad", "i4")])
assert _REQ_DTYPE.itemsize == C.sizeof(rc_request)
assert all(_REQ_DTYPE.fields[n][1] == getattr(rc_request, n).offset for n, _ in rc_request._fields_)


def _ok(st, what):
    if st != RC_OK:
        raise SchedulerError(f"{what} returned {st}")


class Scheduler:
    """Host half of the request lifecycle over a cache object."""

    # slot-row buffers kept for reuse by later native rounds (at most this many)
    ROW_BUFFERS = 4

    def __init__(self, cache, log: list | None = None):
        self.cache = cache
        self.log = log
        self._rows = []

    def _row_buffer(self, n: int) -> np.ndarray:
        """A flat int32 array of n entries for one round's slot rows.  The
        buffer of an earlier round is taken again once nothing refers to it
        any more (every request's slot row is a view that holds a reference),
        so its pages are already mapped: the first write to ~2 MB of fresh
        pages made admission about 3 us per request slower."""
        for b in self._rows:
            # references: the list, the loop variable, getrefcount's argument
            if b.size >= n and sys.getrefcount(b) == 3:
                return b[:n]
        b = np.empty(max(n + n // 8, 1 << 12), np.int32)
        if len(self._rows) >= self.ROW_BUFFERS:
            free = [i for i, x in enumerate(self._rows) if sys.getrefcount(x) == 3]
            if free:
                del self._rows[min(free, key=lambda i: self._rows[i].size)]
        if len(self._rows) < self.ROW_BUFFERS:
            self._rows.append(b)
        return b[:n]

    def _rec(self, *item):
        if self.log is not None:
            self.log.append(item)

    def _native(self) -> bool:
        return self.log is None and hasattr(self.cache, "admit_batch")

    def admit(self, pending: list, policy: int = RC_LPM, max_batch: int | None = None):
        """Admit requests in scheduling order; returns (admitted, still pending)."""
        if not pending:
            return [], []
        if self._native():
            return self._admit_native(pending, policy, max_batch)
        st, order = self.cache.sched_order(policy, [r.prompt for r in pending])
        _ok(st, "sched_order")
        self._rec("order", tuple(int(i) for i in order))
        admitted, waiting = [], []
        blocked = False
        for i in order:
            r = pending[int(i)]
            if blocked or (max_batch is not None and len(admitted) >= max_batch):
                waiting.append(r)
                continue
            st, m, mslots, node = self.cache.match(r.prompt, True)
            _ok(st, "match")
            first = min(m, r.prompt_len - 1) if r.max_new > 0 else m
            need = r.prompt_len - first + r.max_new
            st, new = self.cache.alloc(need)
            self._rec("match", r.rid, m, node, st)
            if st == RC_ERR_NOMEM:
                free = self.cache.stats()["free"]
                est, freed, evlog = self.cache.evict(need - free)
                _ok(est, "evict")
                self._rec("evict", r.rid, need - free, freed, tuple(int(x) for x in evlog))
                st, new = self.cache.alloc(need)
            if st != RC_OK:
                _ok(self.cache.release(node), "release")
                blocked = True
                waiting.append(r)
                self._rec("wait", r.rid)
                continue
            r.node, r.matched, r.first = node, m, first
            r.slots = np.concatenate([mslots[:first], new]).astype(np.int32)
            self._rec("admit", r.rid, tuple(int(x) for x in new[:4]), len(new))
            admitted.append(r)
        # the waiting requests keep their arrival order (the next round's
        # longest-prefix-first order breaks ties by it), as rc_admit's caller does
        took = {id(r) for r in admitted}
        return admitted, [r for r in pending if id(r) not in took]

    # ---- native batch path: the same rules, one C call per round
    def _admit_native(self, pending, policy, max_batch):
        """One rc_admit over a record array filled column by column; the slot
        rows of the round's requests are views into one flat array."""
        n = len(pending)
        req = np.zeros(n, _REQ_DTYPE)
        addr, plen, mnew = [0] * n, [0] * n, [0] * n
        for i, r in enumerate(pending):   # one pass over the requests
            c = getattr(r, "_addr", None)   # Request.tokens_addr's cache
            addr[i] = c[1] if c is not None and c[0] is r.tokens else _tokens_addr(r)
            plen[i], mnew[i] = r.prompt_len, r.max_new
        req["tokens"], req["prompt_len"], req["max_new"] = addr, plen, mnew
        plen, mnew = req["prompt_len"], req["max_new"]
        off = np.zeros(n + 1, np.int64)
        np.cumsum(plen + mnew, out=off[1:])
        flat = self._row_buffer(int(off[-1]))
        req["slots"] = np.uint64(flat.ctypes.data) + 4 * off[:-1].astype(np.uint64)
        order = np.empty(n, np.int32)
        st, cnt = self.cache.admit_batch(policy, req, n, max_batch or 0, order)
        _ok(st, "rc_admit")
        matched, first, node = req["matched"].tolist(), req["first"].tolist(), req["node"].tolist()
        offs = off.tolist()
        rnd = AdmitRound(req, flat, off)
        admitted = []
        for i in order[:cnt].tolist():
            r = pending[i]
            r.matched, r.first, r.node = matched[i], first[i], node[i]
            r.slots = flat[offs[i]:offs[i + 1]]
            r._batch = (rnd, i)
            admitted.append(r)
        if cnt == n:
            return admitted, []
        took = set(order[:cnt].tolist())
        return admitted, [r for i, r in enumerate(pending) if i not in took]

    def _commit_native(self, batch, mode):
        rnd0 = batch[0]._batch[0] if batch else None
        if all(r._batch[0] is rnd0 for r in batch):     # one admission round: one call
            groups = [(rnd0, batch)]
        else:
            by = {}
            for r in batch:
                by.setdefault(id(r._batch[0]), (r._batch[0], []))[1].append(r)
            groups = list(by.values())
        for rnd, rs in groups:
            idx = np.fromiter((r._batch[1] for r in rs), np.int32, len(rs))
            _ok(self.cache.commit_batch(rnd.req, idx, mode), "rc_commit")
            node = rnd.req["node"].tolist()
            for r in rs:
                r.node = node[r._batch[1]]

    def commit_prompts(self, batch: list):
        """After prefill: insert each prompt, keep it pinned, drop the admission pin."""
        if self._native() and all(hasattr(r, "_batch") for r in batch):
            return self._commit_native(batch, RC_COMMIT_PREFILL)
        for r in batch:
            L = r.prompt_len
            st, present, node, canon = self.cache.insert(r.prompt, r.slots[:L], r.max_new > 0)
            _ok(st, "insert")
            self._rec("insert", r.rid, present, node)
            r.slots[:L] = canon
            _ok(self.cache.release(r.node), "release")
            r.node = node if r.max_new > 0 else -1
            if r.max_new == 0:
                self._free_tail(r, L)

    def _free_tail(self, r, n: int):
        """A done request's tokens that the cache did not take (the partial
        last block of a block-granular cache) go back to the pool."""
        tail = getattr(self.cache, "uncached_tail", None)
        k = tail(n) if tail is not None else 0
        if k:
            _ok(self.cache.free(r.slots[n - k:n]), "free")
            self._rec("free_tail", r.rid, k)

    def finish(self, batch: list):
        """After decode: insert prompt + generated tokens, unpin."""
        if self._native() and all(hasattr(r, "_batch") for r in batch):
            return self._commit_native(batch, RC_COMMIT_FINISH)
        for r in batch:
            if r.max_new == 0:
                continue
            n = r.prompt_len + r.max_new
            st, present, node, canon = self.cache.insert(r.tokens[:n], r.slots[:n], False)
            _ok(st, "insert")
            self._rec("finish", r.rid, present, node)
            r.slots[:n] = canon
            _ok(self.cache.release(r.node), "release")
            r.node = -1
            self._free_tail(r, n)


# ------------------------------------------------------------------ cascade
def plan_cascade(rows: list):
    """Shared segments of the batch's cached slot rows (a compressed trie).

    rows[b]: slot ids of row b's positions 0..n_b-1 that other rows may share.
    Returns (segments, private) with segments = [(slots, [row ids])] in the
    order a depth-first walk meets them, and private[b] = the first position of
    row b that no other row shares.
    """
    B = len(rows)
    private = np.zeros(B, np.int64)
    segs = []
    if B == 0:
        return segs, private
    order = sorted(range(B), key=lambda i: rows[i].astype(">i4").tobytes())
    lcp = np.zeros(max(B - 1, 0), np.int64)
    for i in range(B - 1):
        a, b = rows[order[i]], rows[order[i + 1]]
        n = min(len(a), len(b))
        ne = np.flatnonzero(a[:n] != b[:n])
        lcp[i] = ne[0] if ne.size else n
    stack = [(0, B, 0)]
    while stack:
        lo, hi, d = stack.pop()
        if hi - lo == 1:
            private[order[lo]] = d
            continue
        m = int(lcp[lo:hi - 1].min())
        if m > d:
            segs.append((rows[order[lo]][d:m], sorted(order[lo:hi])))
        parts, s = [], lo
        for i in range(lo, hi - 1):
            if lcp[i] == m:
                parts.append((s, i + 1))
                s = i + 1
        parts.append((s, hi))
        for lo2, hi2 in reversed(parts):
            stack.append((lo2, hi2, m))
    return segs, private


def plan_from_rows(rows: list) -> dict:
    """plan_cascade in the dictionary form of rc_cascade_plan."""
    segs, private = plan_cascade(rows)
    B = len(rows)
    if not segs:
        return dict(n_seg=0, private=private)
    seg_rows = np.concatenate([np.asarray(rw, np.int64) for _, rw in segs])
    pos_of = [[] for _ in range(B)]
    for p_, b in enumerate(seg_rows):
        pos_of[int(b)].append(p_)
    return dict(n_seg=len(segs), seg_slots=np.concatenate([sg for sg, _ in segs]).astype(np.int32),
                seg_indptr=np.concatenate([[0], np.cumsum([len(sg) for sg, _ in segs])]).astype(np.int32),
                seg_row_indptr=np.concatenate([[0], np.cumsum([len(rw) for _, rw in segs])]).astype(np.int32),
                seg_rows=seg_rows.astype(np.int32),
                req_seg_indptr=np.concatenate([[0], np.cumsum([len(x) for x in pos_of])]).astype(np.int32),
                req_seg_pos=np.concatenate([np.asarray(x, np.int64) for x in pos_of]).astype(np.int32),
                private=private, max_seg_len=max(len(sg) for sg, _ in segs),
                max_seg_rows=max(len(rw) for _, rw in segs))


# ------------------------------------------------------------------- device
class DeviceEngine:
    """KV pool + slot tables in HBM and the kernel launches of one batch."""

    def __init__(self, shape, pool_slots: int, device="cuda", kv_fp8: bool = False):
        import torch
        self.torch = torch
        self._lib = lib()    # raises if the library is missing
        self.shape = shape
        self.device = torch.device(device)
        self.kv_fp8 = bool(kv_fp8)
        dev = self.device
        self.k_scale = self.v_scale = None
        if shape.mla:
            if kv_fp8:
                raise ValueError("FP8 pools are GQA only")
            self.pool_k = torch.zeros(pool_slots, shape.head_dim_k, dtype=torch.bfloat16, device=dev)
            self.pool_v = None
        elif kv_fp8:  # E4M3 codes and one fp32 scale per (slot, KV head) row
            self.pool_k = torch.zeros(pool_slots, shape.kv_heads, shape.head_dim_k, dtype=torch.uint8, device=dev)
            self.pool_v = torch.zeros(pool_slots, shape.kv_heads, shape.head_dim_v, dtype=torch.uint8, device=dev)
            self.k_scale = torch.zeros(pool_slots, shape.kv_heads, dtype=torch.float32, device=dev)
            self.v_scale = torch.zeros(pool_slots, shape.kv_heads, dtype=torch.float32, device=dev)
        else:
            self.pool_k = torch.zeros(pool_slots, shape.kv_heads, shape.head_dim_k, dtype=torch.bfloat16, device=dev)
            self.pool_v = torch.zeros(pool_slots, shape.kv_heads, shape.head_dim_v, dtype=torch.bfloat16, device=dev)
        self.err = torch.zeros(1, dtype=torch.int32, device=dev)
        self.pool = make_pool_desc(self.pool_k, self.pool_v, self.err, mla=shape.mla, head_dim_v=shape.head_dim_v,
                                   k_scale=self.k_scale, v_scale=self.v_scale)
        self.desc = make_attn_desc(self.pool, shape.q_heads, shape.scale)
        self.sms = torch.cuda.get_device_properties(dev).multi_processor_count if dev.type == "cuda" else 1
        self._ws = torch.zeros(1 << 20, dtype=torch.uint8, device=dev)
        self._stage = [None, None, None]   # [pinned host int32, device int32, event] x 3, used in turn
        self._stage_next = 0
        self._stage_packed = [False] * len(self._stage)   # packed, copy not yet queued
        self._stage_lock = threading.Lock()
        self.pack_wait_s = 0.0       # pack() time blocked on the GPU (on whichever thread packs)
        self.timing = False          # record CUDA events around device calls
        self.timing_every = 1        # decode steps: events on every n-th step only
        self.fuse_store = not kv_fp8  # decode steps store the new token inside attn_decode_append (bf16 pools)
        self.events = {}             # call name -> [(start, end, info)]
        self.launches = 0            # kernels launched by the library (counted per call)
        self.host_wait_s = 0.0       # host time blocked on the GPU (staging buffer reuse)
        self._ev_pool = []

    def start_timing(self, n_events: int = 4096):
        """Record CUDA events around device calls, from a pool made up front
        (each recorded once here, so its CUDA handle exists and the library
        can record it too)."""
        self.events = {}
        self._ev_pool = [self.torch.cuda.Event(enable_timing=True) for _ in range(n_events)]
        for e in self._ev_pool:
            e.record()
        self._ev_next = 0
        self.timing = True

    def _event(self):
        if self._ev_next < len(self._ev_pool):
            e = self._ev_pool[self._ev_next]
            self._ev_next += 1
            return e
        e = self.torch.cuda.Event(enable_timing=True)
        e.record()
        return e

    def _call(self, name, kernels, info, fn):
        if self.timing:
            st = self.torch.cuda.current_stream()
            a = self._event()
            b = self._event()
            a.record(st)
            fn()
            b.record(st)
            self.events.setdefault(name, []).append((a, b, info))
        else:
            fn()
        self.launches += kernels

    def workspace(self, nbytes: int):
        if self._ws.numel() < nbytes:
            self._ws = self.torch.empty(int(nbytes * 1.25) + 256, dtype=self.torch.uint8, device=self.device)
        return self._ws

    def pinned(self, arr):
        """Host array -> pinned host tensor (from torch's caching host allocator,
        which keeps the block until the asynchronous copy that reads it is done)."""
        return self.torch.from_numpy(np.ascontiguousarray(arr)).pin_memory()

    def to_device(self, arr):
        return self.pinned(arr).to(self.device, non_blocking=True)

    def stage(self, arrays: list) -> list:
        """Host int32 arrays -> device, through one pinned staging buffer and
        one host-to-device copy; returns device views in the same order and
        shapes (pack() then upload())."""
        ticket = self.pack(arrays)
        self.host_wait_s += ticket[3]
        return self.upload(ticket)

    def pack(self, arrays: list):
        """Host half of stage(): the arrays packed into the next pinned
        staging buffer (256-byte aligned views).  May run on another thread
        than upload(); each ticket must be uploaded before two more are
        packed.  A buffer is rewritten only after the copy that last read it
        has run (host wait counted in pack_wait_s)."""
        torch = self.torch
        offs, n = [], 0
        for a in arrays:
            offs.append(n)
            n += (a.size + 63) // 64 * 64
        n = max(n, 64)
        with self._stage_lock:
            k = self._stage_next
            self._stage_next = (k + 1) % len(self._stage)
            if self._stage_packed[k]:
                raise RuntimeError("staging buffer packed twice without an upload")
            self._stage_packed[k] = True
        slot = self._stage[k]
        waited = 0.0
        if slot is None:
            slot = self._stage[k] = [None, None, torch.cuda.Event()]
        else:
            t0 = time.perf_counter()
            slot[2].synchronize()
            waited = time.perf_counter() - t0
            self.pack_wait_s += waited
        if slot[0] is None or slot[0].numel() < n:   # (the device half grows in upload())
            slot[0] = torch.empty(max(n + n // 4, 1 << 16), dtype=torch.int32).pin_memory()
        hv = slot[0].numpy()
        for a, o in zip(arrays, offs):
            hv[o:o + a.size] = a.reshape(-1)
        return k, n, [(o, a.size, a.shape) for a, o in zip(arrays, offs)], waited

    def upload(self, ticket) -> list:
        """Device half of stage(): one host-to-device copy of a packed buffer,
        ordered on the current stream after every earlier kernel (so kernels
        of an earlier batch have finished reading the device buffer it
        overwrites); returns the device views."""
        k, n, views, _ = ticket
        slot = self._stage[k]
        if slot[1] is None or slot[1].numel() < n:
            slot[1] = self.torch.empty(slot[0].numel(), dtype=self.torch.int32, device=self.device)
        host, dev, ev = slot
        dev[:n].copy_(host[:n], non_blocking=True)
        ev.record()
        with self._stage_lock:
            self._stage_packed[k] = False
        return [dev[o:o + size].view(shape) for o, size, shape in views]

    def upload_batch(self, batch: list, cascade: bool, planner=None, parts=("extend", "decode")):
        """Slot rows and index arrays of the batch -> device; returns its layout."""
        return BatchLayout(self, batch, cascade, planner, parts)

    # -- kernels
    def store(self, slots_dev, k, v):
        n = int(slots_dev.numel())
        if n:
            self._call("kv_store", 1, ("store", n), lambda: kv_store(self.pool, slots_dev, k, v))

    def extend(self, lay, q, out, lse=None):
        kv = lay.extend_table
        self._call("attn_extend", 1, ("extend", lay),
                   lambda: attn_extend(self.desc, q, lay.qo_indptr, kv, lay.batch_size, lay.max_q, out, lse))

    # ---- decode loop: per-step arguments built once per batch, two C calls per step
    def prepare_decode(self, lay):
        T, B = lay.max_new, lay.batch_size
        casc = lay.casc if lay.use_cascade else None
        lay.kv_tables = None
        dec_max = lay.dec_max.tolist() if T else []
        # the workspace attn_decode plans grows with max_len: size it for the largest
        lay.ws_bytes = self._decode_ws(B, [max(dec_max)] if dec_max else [], casc)
        lay.ws = self.workspace(lay.ws_bytes)
        lay.ws_ptr = lay.ws.data_ptr()
        lay.casc_ref = C.byref(casc) if casc is not None else None
        # step t's rows of the [T, B] int32 arrays: base + 4 B t (no per-step tensor views)
        if T:
            assert lay.decode_slots.is_contiguous() and lay.dec_len.is_contiguous()
        p0 = lay.decode_slots.data_ptr() if T else 0
        lay.slot_ptrs = [p0 + 4 * B * t for t in range(T)]
        # one table descriptor, its length row and bound set per step
        lay.kv = make_kv_table(lay.table, lay.dec_start, lay.dec_len[0], dec_max[0]) if T else None
        lay.kv_ref = C.byref(lay.kv) if T else None
        p0 = lay.dec_len.data_ptr() if T else 0
        lay.len_ptrs = [p0 + 4 * B * t for t in range(T)]
        lay.dec_max_list = dec_max
        lay.pool_ref = C.byref(self.pool)
        lay.desc_ref = C.byref(self.desc)
        # kernels per step: cascade (if any) + table pass + merge when a row is split
        # (the same thresholds as the library's plan)
        sms = self.sms
        if self.shape.mla:
            max_len = max(dec_max) if dec_max else 0
            if self.shape.q_heads == 128:   # tcgen05 latent kernel: chunks of 256..4096 keys
                c = max(256, min(4096, -(-(B * max_len // (4 * sms)) // 32) * 32)) if max_len else 32
                split = max_len > c
            else:
                base = B * (self.shape.q_heads // 16)
                splits = min(max(-(-4 * sms // max(base, 1)), 1), max(-(-max_len // 1024), 1))
                split = splits > 1
        else:
            split = B * self.shape.kv_heads < 8 * sms
        lay.decode_kernels = (1 if casc is not None else 0) + 1 + (1 if split else 0)
        lay.stream = C.c_void_p(self.torch.cuda.current_stream(self.device).cuda_stream)
        lay.step_arr = None

    def _decode_ws(self, B: int, max_lens, casc) -> int:
        """Largest workspace attn_decode asks for over the steps' bounds."""
        L = lib()
        dref = C.byref(self.desc)
        cref = C.byref(casc) if casc is not None else None
        n = C.c_size_t(0)
        best = 256
        for m in max_lens:
            st = L.attn_decode_workspace(dref, B, int(m), cref, C.byref(n))
            if st != RC_OK:
                raise RCError("attn_decode_workspace", st)
            best = max(best, n.value)
        return best

    def decode_step(self, lay, t: int, q, k, v, out, lse=None):
        """One decode step: the new token's K/V goes into its slot and the
        step's attention runs -- fused into one call (attn_decode_append)
        for GQA pools, kv_store + attn_decode for the latent layout."""
        L = self._lib
        B = lay.batch_size
        ev = None
        if self.timing and t % self.timing_every == 0:
            ev = (self._event(), self._event())
            ev[0].record()
        kv = lay.kv
        kv.len = lay.len_ptrs[t]          # read by the call itself, not by its kernels
        kv.max_len = lay.dec_max_list[t]
        if self.fuse_store and v is not None:
            st = L.attn_decode_append(lay.desc_ref, q.data_ptr(), k.data_ptr(), v.data_ptr(), lay.kv_ref, B,
                                      lay.casc_ref, out.data_ptr(), lse.data_ptr() if lse is not None else None,
                                      lay.ws_ptr, lay.ws_bytes, lay.stream)
            if st != RC_OK:
                raise RCError("attn_decode_append", st)
            kernels = lay.decode_kernels
        else:
            st = L.kv_store(lay.pool_ref, lay.slot_ptrs[t], k.data_ptr(), v.data_ptr() if v is not None else None,
                            B, None, None, lay.stream)
            if st != RC_OK:
                raise RCError("kv_store", st)
            st = L.attn_decode(lay.desc_ref, q.data_ptr(), lay.kv_ref, B, lay.casc_ref,
                               out.data_ptr(), lse.data_ptr() if lse is not None else None, lay.ws.data_ptr(),
                               lay.ws_bytes, lay.stream)
            if st != RC_OK:
                raise RCError("attn_decode", st)
            kernels = 1 + lay.decode_kernels
        if ev:
            ev[1].record()
            self.events.setdefault("attn_decode", []).append((ev[0], ev[1], ("decode", lay, t)))
        self.launches += kernels

    def decode_steps(self, lay, t0: int, ins, outs, lses=None):
        """Decode steps t0 .. t0+n-1 of the batch in one library call
        (attn_decode_steps): the launches decode_step makes for each step,
        in the same order, queued by one C call (inside a run, a step's
        cascade reads before the previous step's table pass has finished).
        ins[i]: step t0+i's q/k/v; outs[i], lses[i]: where it writes.  With
        timing on, one pair of CUDA events spans the whole run (events between
        steps would hold each cascade back until the previous step ends)."""
        n = len(ins)
        arr = lay.step_arr
        if arr is None or len(arr) < n:
            arr = lay.step_arr = (rc_decode_step * max(n, 16))()
        fused = self.fuse_store
        timed = []
        for i in range(n):
            t = t0 + i
            inp, a = ins[i], arr[i]
            k, v = inp["k"], inp["v"]
            a.q = inp["q"].data_ptr()
            a.out = outs[i].data_ptr()
            a.lse = lses[i].data_ptr() if lses is not None else None
            a.len = lay.len_ptrs[t]
            a.max_len = lay.dec_max_list[t]
            a.k_new = k.data_ptr()
            a.v_new = v.data_ptr() if v is not None else None
            a.store_slots = None if fused and v is not None else lay.slot_ptrs[t]
            a.ev_begin = a.ev_end = None
        if self.timing:
            e0, e1 = self._event(), self._event()
            arr[0].ev_begin, arr[n - 1].ev_end = e0.cuda_event, e1.cuda_event
            timed.append((e0, e1, ("decode", lay, t0, n)))
        st = self._lib.attn_decode_steps(lay.desc_ref, lay.kv_ref, lay.batch_size, lay.casc_ref, arr, n,
                                         lay.ws_ptr, lay.ws_bytes, lay.stream, None)
        if st != RC_OK:
            raise RCError("attn_decode_steps", st)
        if timed:
            self.events.setdefault("attn_decode", []).extend(timed)
        per = lay.decode_kernels if fused and ins[0]["v"] is not None else 1 + lay.decode_kernels
        self.launches += n * per

    def decode(self, lay, t: int, q, out, lse=None):
        kv, casc = lay.decode_table(t)
        ws_bytes = attn_decode_workspace(self.desc, lay.batch_size, kv.max_len, casc)
        ws = self.workspace(ws_bytes)
        self._call("attn_decode", 3 if casc is not None else 2, ("decode", lay, t),
                   lambda: attn_decode(self.desc, q, kv, lay.batch_size, out, lse, ws, cascade=casc))


class BatchLayout:
    """Device-side index arrays of one admitted batch (one staging copy).

    parts: "extend" (prefill: new-token slots, per-request extents) and/or
    "decode" (per-step slots and lengths, cascade segments).  A batch taken
    from one native admission round is laid out from the round's flat slot
    array with vectorised indexing; otherwise from each request's slot row."""

    def __init__(self, eng: DeviceEngine, batch: list, cascade: bool, planner=None,
                 parts=("extend", "decode"), defer: bool = False):
        """defer=True stops after the host arrays are packed into a staging
        buffer (eng.pack: it may run on a worker thread); upload() then
        queues the copy and sets the device views."""
        self.eng = eng
        self.batch = batch
        self.batch_size = B = len(batch)
        rnd = batch[0]._batch[0] if B and hasattr(batch[0], "_batch") else None
        if rnd is not None and all(getattr(r, "_batch", (None,))[0] is rnd for r in batch):
            idx = np.fromiter((r._batch[1] for r in batch), np.int64, B)
            flat = rnd.flat
            starts = rnd.off[idx]
            L = rnd.req["prompt_len"][idx]
            first = rnd.req["first"][idx]
            max_new = rnd.req["max_new"][idx]
        else:
            rows = np.fromiter((len(r.slots) for r in batch), np.int64, B)
            starts = np.zeros(B, np.int64)
            if B > 1:
                np.cumsum(rows[:-1], out=starts[1:])
            flat = np.concatenate([r.slots for r in batch]) if B else np.zeros(0, np.int32)
            L = np.fromiter((r.prompt_len for r in batch), np.int64, B)
            first = np.fromiter((r.first for r in batch), np.int64, B)
            max_new = np.fromiter((r.max_new for r in batch), np.int64, B)
        n_new = L - first
        self.L, self.first, self.starts = L, first, starts
        self.max_new = int(max_new.max()) if B else 0
        qo = np.zeros(B + 1, np.int64)
        np.cumsum(n_new, out=qo[1:])
        self.qo_host = qo
        self.max_q = int(n_new.max()) if B else 0
        host = [flat, starts, L]
        names = ["table", "start_dev", "len_prompt"]
        if "extend" in parts:
            # slots of new tokens, in (request, position) order
            pos = np.repeat(starts + first - qo[:-1], n_new) + np.arange(int(qo[-1]))
            host += [qo, flat[pos]]
            names += ["qo_indptr", "extend_slots"]
        self.use_cascade = False
        self.private = np.zeros(B, np.int64)
        self.casc = None
        plan = None
        T = self.max_new if "decode" in parts else 0
        if T:
            if (max_new != T).any():
                raise ValueError("a decode batch needs one max_new for all its requests")
            # slots of step t for every row [T, B], and per-step lengths
            dec = flat[(starts + L)[None, :] + np.arange(T)[:, None]]
            lens = L[None, :] + np.arange(T)[:, None] + 1
            self.use_cascade = cascade and B > 1
            if self.use_cascade:
                if planner is not None and all(r.node >= 0 for r in batch):
                    plan = planner(np.fromiter((r.node for r in batch), np.int64, B))   # read off the tree
                else:
                    plan = plan_from_rows([r.slots[:r.prompt_len] for r in batch])
                if plan["n_seg"] > 0:
                    self.private = plan["private"].astype(np.int64)
                    ip = plan["seg_indptr"]
                    self.segments = [(plan["seg_slots"][ip[k]:ip[k + 1]],
                                      plan["seg_rows"][plan["seg_row_indptr"][k]:plan["seg_row_indptr"][k + 1]])
                                     for k in range(plan["n_seg"])]
                else:
                    self.use_cascade = False
                    plan = None
            dec_len = lens - self.private[None, :]
            self.dec_max = dec_len.max(axis=1)
            host += [dec, starts + self.private, dec_len]
            names += ["decode_slots", "dec_start", "dec_len"]
        else:
            self.dec_max = None
        casc_keys = ("seg_slots", "seg_indptr", "seg_row_indptr", "seg_rows", "req_seg_indptr", "req_seg_pos")
        if plan is not None:
            host += [np.asarray(plan[k]) for k in casc_keys]
        host = [np.asarray(a, np.int32) for a in host]
        self._names, self._plan, self._T, self._parts = names, plan, T, parts
        self._ticket = None
        if defer:
            self._ticket = eng.pack(host)
        else:
            self._set_device(eng.stage(host))

    def upload(self):
        """The deferred half: the packed arrays' copy and the device views."""
        self._set_device(self.eng.upload(self._ticket))
        self._ticket = None
        return self

    def _set_device(self, dv):
        names, plan, T, parts = self._names, self._plan, self._T, self._parts
        B, L = self.batch_size, self.L
        for nm, t in zip(names, dv):
            setattr(self, nm, t)
        if "extend" not in parts:
            self.qo_indptr = self.extend_slots = None
        if not T:
            self.decode_slots = self.dec_start = self.dec_len = None
        if plan is not None:
            self._casc_arrays = dv[len(names):]
            self.casc = make_cascade(*self._casc_arrays, max_seg_rows=plan["max_seg_rows"],
                                     max_seg_len=plan["max_seg_len"], host_seg_indptr=plan["seg_indptr"],
                                     host_seg_row_indptr=plan["seg_row_indptr"])
        self.extend_table = make_kv_table(self.table, self.start_dev, self.len_prompt, int(L.max()) if B else 0)

    def decode_table(self, t: int):
        kv = make_kv_table(self.table, self.dec_start, self.dec_len[t], int(self.dec_max[t]))
        return kv, (self.casc if self.use_cascade else None)
