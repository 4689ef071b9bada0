"""Host-side request traces run through any cache object (oracle tree or product).

Every call's result goes into a log, so two implementations can be compared
result by result.
"""
from __future__ import annotations

import numpy as np

OK, NOMEM = 0, -2


def serve_prefill(cache, prompt, log=None):
    """One prefill-only request, run alone: match+pin, allocate (evicting if
    needed), insert, unpin.  Returns the matched length, or -1 if it could not fit."""
    st, m, mslots, node = cache.match(prompt, True)
    assert st == OK
    need = len(prompt) - m
    st, new = cache.alloc(need)
    ev = None
    if st == NOMEM:
        free = cache.stats()["free"]
        est, freed, evlog = cache.evict(need - free)
        assert est == OK
        ev = (need - free, freed, tuple(int(x) for x in evlog))
        st, new = cache.alloc(need)
    if st != OK:
        assert cache.release(node) == OK
        if log is not None:
            log.append(("nofit", m, ev))
        return -1
    slots = np.concatenate([mslots, new]).astype(np.int32)
    st, present, node2, canon = cache.insert(prompt, slots, False)
    assert st == OK and present == m
    assert cache.release(node) == OK
    if log is not None:
        log.append(("served", m, node, node2, ev, tuple(int(x) for x in new[:8])))
    return m


def cyclic_hits(cache_factory, prefixes, order, pool):
    cache = cache_factory(pool)
    hits = 0
    for p in order:
        m = serve_prefill(cache, prefixes[p])
        hits += m > 0
    return hits


def run_batch_sequential(cache, prompts, order, log=None):
    """Serve prompts one at a time in the given order; returns total matched tokens."""
    total = 0
    for i in order:
        m = serve_prefill(cache, prompts[i], log)
        assert m >= 0
        total += m
    return total


def lpm_dynamic_order(cache, prompts):
    """Longest-cached-prefix-first, re-evaluated after every request (one at a time)."""
    pending = list(range(len(prompts)))
    total = 0
    while pending:
        st, order = cache.sched_order(1, [prompts[i] for i in pending])
        assert st == OK
        i = pending.pop(int(order[0]))
        total += serve_prefill(cache, prompts[i])
    return total


def random_trace(cache, rng, n_ops, vocab=4, max_len=12, log=None, bases=None):
    """Random mix of every host call over a tiny vocabulary (forces splits,
    duplicates, evictions, pinning errors).  Logs every result.  With `bases`
    (token arrays), most requests are a prefix of one of them, possibly with
    one token changed, so that long shared prefixes occur."""
    pinned = []      # node handles we hold pins on
    held = []        # slots we own
    for _ in range(n_ops):
        op = rng.integers(0, 7)
        if op in (0, 1):  # request: match+pin, alloc, insert (pin or not), maybe release
            n = int(rng.integers(1, max_len + 1))
            tok = rng.integers(0, vocab, n).astype(np.int32)
            if bases is not None and rng.random() < 0.8:
                base = bases[int(rng.integers(0, len(bases)))]
                n = min(n, len(base))
                tok = base[:n].copy()
                if rng.random() < 0.3:
                    tok[int(rng.integers(0, n))] = int(rng.integers(0, vocab))
            st, m, ms, node = cache.match(tok, True)
            log.append(("match", st, m, tuple(int(x) for x in ms), node))
            st, new = cache.alloc(n - m)
            log.append(("alloc", st, tuple(int(x) for x in new)))
            if st != OK:
                log.append(("rel", cache.release(node)))
                continue
            slots = np.concatenate([ms, new]).astype(np.int32)
            mine = [int(x) for x in new]
            if rng.random() < 0.3 and m > 0:  # recompute a few cached tokens: duplicates
                k = int(rng.integers(1, m + 1))
                st, extra = cache.alloc(k)
                log.append(("alloc", st, tuple(int(x) for x in extra)))
                if st == OK:
                    slots[m - k:m] = extra
                    mine += [int(x) for x in extra]
            pin = bool(rng.integers(0, 2))
            st, present, node2, canon = cache.insert(tok, slots, pin)
            log.append(("insert", st, present, node2, tuple(int(x) for x in canon)))
            if st != OK:
                held.extend(mine)
            elif hasattr(cache, "uncached_tail"):  # a block cache leaves the partial block with us
                k = cache.uncached_tail(n)
                held.extend(int(x) for x in canon[n - k:])
            log.append(("rel", cache.release(node)))
            if pin and st == OK:
                pinned.append(node2)
        elif op == 2 and pinned:
            i = int(rng.integers(0, len(pinned)))
            log.append(("rel", cache.release(pinned.pop(i))))
        elif op == 3:
            st, freed, ev = cache.evict(int(rng.integers(0, 16)))
            log.append(("evict", st, freed, tuple(int(x) for x in ev)))
        elif op == 4:
            n = int(rng.integers(0, 8))
            st, s = cache.alloc(n)
            log.append(("alloc", st, tuple(int(x) for x in s)))
            if st == OK:
                held.extend(int(x) for x in s)
        elif op == 5 and held:
            k = int(rng.integers(1, len(held) + 1))
            give = held[:k]
            st = cache.free(np.asarray(give, np.int32))
            log.append(("free", st))
            if st == OK:
                del held[:k]
        elif op == 6:
            prompts = [rng.integers(0, vocab, int(rng.integers(0, max_len))).astype(np.int32) for _ in range(4)]
            st, order = cache.sched_order(int(rng.integers(0, 2)), prompts)
            log.append(("order", st, tuple(int(x) for x in order)))
            # error paths: unknown node, double release, bad slot ids
            log.append(("bad_rel", cache.release(10 ** 9)))
            log.append(("bad_free", cache.free(np.asarray([-1], np.int32))))
        log.append(("stats", tuple(sorted(cache.stats().items()))))
    return log
