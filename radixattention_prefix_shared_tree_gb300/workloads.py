"""Serving loops of the five workloads over the driver.

``Runner.serve`` is one scheduling round of continuous batching: admit (in
``sched_order`` order, evicting as needed), prefill the admitted batch
(kv_store of the new tokens, attn_extend), insert the prompts, decode every
step (kv_store + attn_decode, flat or cascade), insert prompt + outputs and
unpin.  Without a device engine only the host calls run (used to replay a
workload through two cache implementations).  The model object supplies
token sequences and Q/K/V rows; the workload shapes come from the caller.
"""
from __future__ import annotations

import time

import numpy as np

from . import RC_LPM
from .driver import Request, Scheduler


def new_request(model, rid: int, prompt, max_new: int) -> Request:
    toks, hashes = model.sequence(np.asarray(prompt, np.int32), max_new)
    model.register(rid, hashes)
    r = Request(rid=rid, tokens=toks, prompt_len=len(prompt), max_new=max_new)
    r.tokens_addr()   # taken once, at intake, rather than in every admission round
    return r


class Runner:
    def __init__(self, cache, model, engine=None, policy: int = RC_LPM, cascade: bool = True,
                 collect: bool = False, prefill_attention: bool = True, log: list | None = None,
                 sched=None):
        # sched: any object with admit / commit_prompts / finish (default: the
        # driver's Scheduler over `cache`)
        self.sched = sched if sched is not None else Scheduler(cache, log)
        self.cache = cache
        self.model = model
        self.engine = engine
        self.policy = policy
        self.cascade = cascade
        self.collect = collect
        self.prefill_attention = prefill_attention
        self.extend_out = {}   # rid -> (positions, out bf16 [n, Hq, dv], lse [n, Hq])
        self.decode_out = {}   # rid -> list of (position, out [Hq, dv], lse [Hq])
        self.next_rid = 0
        self.collect_rids = None  # collect only these requests' outputs (None: all)
        self.on_decode = None   # optional callback(out, t, n_steps) after each decode step
        self.on_extend = None   # optional callback(out) after the prefill
        self.decode_out_slots = 1  # decode step t writes slot t mod this of `decode_outs`
        self.decode_chunk = 16     # decode steps queued per library call
        self.decode_outs = None
        self.worker_wait_s = 0.0   # overlapped rounds: time this thread waited for the worker

    def request(self, prompt, max_new: int) -> Request:
        r = new_request(self.model, self.next_rid, prompt, max_new)
        self.next_rid += 1
        return r

    # ------------------------------------------------------------ one round
    def serve(self, pending: list, max_batch: int | None = None):
        admitted, waiting = self.sched.admit(pending, self.policy, max_batch)
        if admitted:
            if self.engine is not None:
                self._prefill(admitted)
            self.sched.commit_prompts(admitted)
            if self.engine is not None and any(r.max_new for r in admitted):
                self._decode([r for r in admitted if r.max_new])
            self.sched.finish(admitted)
        return admitted, waiting

    # -------------------------------------------------------- many rounds
    def serve_rounds(self, pending: list, after, max_batch: int | None = None, overlap: bool = False):
        """Rounds of continuous batching: serve `pending`, then
        after(admitted, waiting) gives the next round's queue (None: done).

        overlap=True is the overlapped scheduler (the SGLang engineering
        article's zero-overhead batch scheduler, section 2: the CPU prepares
        batch k+1 while the GPU runs batch k).  Round k's finish inserts,
        then round k+1's whole admission (order, match, pin, evict, alloc),
        its prompt inserts and its index arrays (slot table, cascade plan,
        packed into a pinned staging buffer) are made on a worker thread
        while this thread launches round k's decode steps; the native calls
        release the interpreter lock, so the two overlap.  The tree sees the
        same calls in the same order as serve() round by round (the launches
        touch no tree state, and every kernel of round k+1 is queued after
        round k's on the one stream, so slots round k+1 takes from round k
        are written only after round k has read them).  A round's prompts
        are inserted before its prefill is queued rather than after: a
        prompt part another request inserted first then maps to that
        request's slots, which the prefill fills with the same K/V (a
        deterministic function of the tokens), so the results are
        identical."""
        if not overlap:
            while pending:
                admitted, waiting = self.serve(pending, max_batch)
                pending = after(admitted, waiting)
            return
        from concurrent.futures import ThreadPoolExecutor
        sched, policy = self.sched, self.policy

        def admit_commit(queue):
            admitted, waiting = sched.admit(queue, policy, max_batch)
            ready = None
            if admitted:
                sched.commit_prompts(admitted)
                if self.engine is not None and self._one_layout(admitted):
                    ready = self._round_layout(admitted, defer=True)   # packed here, uploaded by the caller
            return admitted, waiting, ready

        with ThreadPoolExecutor(1) as worker:
            fut = worker.submit(admit_commit, pending)
            while True:
                t_wait = time.perf_counter()
                admitted, waiting, ready = fut.result()
                self.worker_wait_s += time.perf_counter() - t_wait
                nxt = after(admitted, waiting)
                lay = None
                if admitted and self.engine is not None:
                    dec = [r for r in admitted if r.max_new]
                    ext = None
                    if ready is not None:
                        ext = self.last_layout = ready.upload()
                    self._prefill(admitted, ext)
                    if dec:   # (a decode layout reads the tree: before the worker goes on)
                        lay = ext if ext is not None else self._decode_layout(dec)

                def host_work(admitted=admitted, nxt=nxt):
                    if admitted:
                        sched.finish(admitted)
                    return admit_commit(nxt) if nxt else ([], [], None)
                fut = worker.submit(host_work)
                if lay is not None:
                    self._decode_steps(dec, lay)
                if not nxt:
                    t_wait = time.perf_counter()
                    fut.result()
                    self.worker_wait_s += time.perf_counter() - t_wait
                    return

    def _prefill(self, batch, lay=None):
        eng, torch = self.engine, self.engine.torch
        if lay is None:
            lay = eng.upload_batch(batch, cascade=False, parts=("extend",))
        total = int(lay.qo_host[-1])
        if total == 0:
            return
        if not self.prefill_attention:   # store K/V only (no queries needed)
            inp = self.model.extend_kv(batch)
            eng.store(lay.extend_slots, inp["k"], inp["v"])
            return
        inp = self.model.extend_inputs(batch)
        eng.store(lay.extend_slots, inp["k"], inp["v"])
        sh = eng.shape
        out = torch.empty(total, sh.q_heads, sh.head_dim_v, dtype=torch.bfloat16, device=eng.device)
        lse = torch.empty(total, sh.q_heads, dtype=torch.float32, device=eng.device) if self.collect else None
        eng.extend(lay, inp["q"], out, lse)
        if self.on_extend is not None:
            self.on_extend(out)
        if self.collect:
            for i, r in enumerate(batch):
                if self.collect_rids is not None and r.rid not in self.collect_rids:
                    continue
                a, b = int(lay.qo_host[i]), int(lay.qo_host[i + 1])
                o = out[a:b].view(torch.int16).cpu().numpy().view(np.uint16)
                self.extend_out[r.rid] = (np.arange(r.first, r.prompt_len), o, lse[a:b].cpu().numpy())

    def _decode(self, batch):
        self._decode_steps(batch, self._decode_layout(batch))

    def _decode_layout(self, batch):
        """Slot tables and cascade segments of a decode batch, staged to the
        device (the cascade plan is read off the tree's pinned paths)."""
        planner = getattr(self.cache, "cascade_plan", None)
        lay = self.engine.upload_batch(batch, cascade=self.cascade, planner=planner, parts=("decode",))
        self.last_layout = lay
        return lay

    @staticmethod
    def _one_layout(batch) -> bool:
        """Every request decodes, the same number of tokens: one layout
        serves the round's prefill and its decode steps."""
        return all(r.max_new for r in batch) and len({r.max_new for r in batch}) == 1

    def _round_layout(self, batch, defer: bool = False):
        """One layout for the prefill and the decode steps of a round
        (_one_layout), laid out after the round's prompt inserts so the slot
        table is staged once instead of once per phase.  defer=True: host
        arrays packed, BatchLayout.upload() left to the launching thread."""
        from .driver import BatchLayout
        planner = getattr(self.cache, "cascade_plan", None)
        return BatchLayout(self.engine, batch, self.cascade, planner, ("extend", "decode"), defer=defer)

    def _decode_steps(self, batch, lay):
        """Every decode step of the batch, in runs of up to `decode_chunk`
        steps (aligned to multiples of it), each run queued by one library
        call (attn_decode_steps); decode_chunk = 1 makes one decode_step call
        per step.  Step t writes slot t mod R of `decode_outs`."""
        eng, torch = self.engine, self.engine.torch
        sh = eng.shape
        B, T = len(batch), lay.max_new
        CH = max(1, self.decode_chunk)
        R = max(1, self.decode_out_slots)
        if self.collect:
            R = max(R, CH)     # a run's outputs are read after the run
        outs = torch.empty(R, B, sh.q_heads, sh.head_dim_v, dtype=torch.bfloat16, device=eng.device)
        self.decode_outs = outs
        views = [outs[i] for i in range(R)]
        lses = None
        idx = None
        if self.collect:
            ring = torch.empty(R, B, sh.q_heads, dtype=torch.float32, device=eng.device)
            lses = [ring[i] for i in range(R)]
            if self.collect_rids is None:
                idx = list(range(B))
            else:
                idx = [i for i, r in enumerate(batch) if r.rid in self.collect_rids]
            sel = torch.as_tensor(idx, device=eng.device) if idx else None
        eng.prepare_decode(lay)
        t = 0
        while t < T:
            n = min(CH - t % CH, T - t)
            ins = [self.model.decode_inputs(batch, t + i) for i in range(n)]
            ov = [views[(t + i) % R] for i in range(n)]
            lv = [lses[(t + i) % R] for i in range(n)] if lses is not None else None
            if CH == 1:
                inp = ins[0]
                eng.decode_step(lay, t, inp["q"], inp["k"], inp["v"], ov[0], lv[0] if lv else None)
            else:
                eng.decode_steps(lay, t, ins, ov, lv)
            for i in range(n):
                if self.on_decode is not None:
                    self.on_decode(ov[i], t + i, T)
                if idx:
                    o = ov[i].index_select(0, sel).view(torch.int16).cpu().numpy().view(np.uint16)
                    l = lv[i].index_select(0, sel).cpu().numpy()
                    for j, b in enumerate(idx):
                        self.decode_out.setdefault(batch[b].rid, []).append((batch[b].prompt_len + t + i, o[j], l[j]))
            t += n


# ------------------------------------------------------------------ workloads
def run_tiny(runner: Runner, trace):
    """Requests one at a time: prefill, decode max_new tokens, finish."""
    reqs = []
    for p in trace.prompts:
        r = runner.request(p, trace.max_new)
        admitted, waiting = runner.serve([r])
        assert admitted and not waiting
        reqs.append(r)
    return reqs


def run_cyclic(runner: Runner, prefixes, order):
    """Prefill-only requests one at a time; returns the number of hits."""
    hits = 0
    for p in order:
        r = runner.request(prefixes[p], 0)
        admitted, _ = runner.serve([r])
        assert admitted
        hits += r.matched > 0
    return hits


def run_few_shot(runner: Runner, trace, warm: bool = True):
    """The shared examples once (prefill only), then all questions in one batch."""
    if warm:
        runner.serve([runner.request(trace.warm, 0)])
    reqs = [runner.request(trace.prompt(i), trace.max_new) for i in range(len(trace.questions))]
    admitted, waiting = runner.serve(reqs)
    assert not waiting
    return admitted


def run_chat(runner: Runner, trace, max_rounds: int = 10_000, overlap: bool = False):
    """Sessions grow turn by turn; each round admits the ready turns that fit."""
    n_sess = len(trace.user_turns)
    history = [np.zeros(0, np.int32) for _ in range(n_sess)]
    turn = [0] * n_sess
    pending = {}
    for s in range(n_sess):
        r = runner.request(trace.user_turns[s][0], trace.max_new)
        r.session = s
        pending[s] = r
    served = []
    rounds = [0]

    def after(admitted, waiting):
        rounds[0] += 1
        if not admitted:
            raise RuntimeError("no progress: pool too small for any waiting turn")
        for r in admitted:
            s = r.session
            served.append(r)
            history[s] = r.tokens[:r.prompt_len + r.max_new]
            turn[s] += 1
            del pending[s]
            if turn[s] < len(trace.user_turns[s]):
                nr = runner.request(np.concatenate([history[s], trace.user_turns[s][turn[s]]]), trace.max_new)
                nr.session = s
                pending[s] = nr
        if not pending or rounds[0] >= max_rounds:
            return None
        return [pending[s] for s in sorted(pending)]

    runner.serve_rounds([pending[s] for s in sorted(pending)], after, trace.max_batch, overlap)
    return served, rounds[0]


def run_agent(runner: Runner, trace, overlap: bool = False):
    """Root prompt, then each level of branches (prefill only), then all leaves decode."""
    depth = len(trace.leaves[0])
    levels = [[trace.root]] + [[trace.prompt(p) for p in sorted({leaf[:lvl] for leaf in trace.leaves})]
                               for lvl in range(1, depth)]
    out = []

    def after(admitted, waiting):
        assert not waiting
        out[:] = admitted
        if levels:
            return [runner.request(p, 0) for p in levels.pop(0)]
        if out and out[0].max_new == 0 and not getattr(after, "leaves_done", False):
            after.leaves_done = True
            return [runner.request(trace.prompt(leaf), trace.max_new) for leaf in trace.leaves]
        return None

    first = [runner.request(p, 0) for p in levels.pop(0)]
    runner.serve_rounds(first, after, None, overlap)
    return out


def run_mla(runner: Runner, trace, n_requests: int | None = None, overlap: bool = False):
    """Latent-attention long-context decode: the shared prefix and every
    request's private context are stored (kv_store, no prefill attention),
    then all requests decode trace.steps tokens together."""
    n = len(trace.private) if n_requests is None else n_requests
    out = []
    todo = [lambda: [runner.request(trace.prompt(i), trace.steps) for i in range(n)]]

    def after(admitted, waiting):
        assert not waiting
        out[:] = admitted
        return todo.pop(0)() if todo else None

    runner.serve_rounds([runner.request(trace.shared, 0)], after, None, overlap)
    return out


def run_multimodal(runner: Runner, trace, key_fn, batch: int = 64, overlap: bool = False):
    """Questions about images in arrival order, served in rounds of up to
    `batch` (the scheduler orders each round); an image's key run comes from
    key_fn(bytes, n_tokens)."""
    reqs = [runner.request(trace.prompt(i, key_fn), trace.max_new) for i in range(len(trace.questions))]
    served = []

    def after(admitted, waiting):
        if not admitted:
            raise RuntimeError("no progress: pool too small for any waiting request")
        served.extend(admitted)
        return waiting or None

    runner.serve_rounds(reqs, after, batch, overlap)
    return served
