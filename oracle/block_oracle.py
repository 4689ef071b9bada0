"""Oracle of the block-granular comparator cache and of image keys: test
infrastructure.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this module.  It shares no code with the product library.

Block cache -- "RadixAttention, eviction and cache churn" (inference-notes
note 49), section 3: vLLM keeps each 16-token block under a hash chain of the
prefix, matches whole blocks only, shares blocks by reference count and evicts
the least recently used first.  The readings (the section gives a table, not
rules in detail) are the product's, stated in its header: only full blocks
are cached, keyed exactly by (the block before, its tokens); a lookup walks
whole blocks from the start; insert caches the full blocks not cached yet and
the partial last block stays with the caller; every match and insert advance
a clock by one and stamp the chain (root included); pins count per block of
the chain; eviction takes unpinned blocks (never the root) in order of
(last access, farther from the chain's start first, id), whole blocks, until
the freed count reaches the request; the allocator gives the n smallest free
ids.  Written plainly: a dict of blocks, a sorted free list, a full scan for
each eviction victim.

Image keys -- the unite.ai article on SGLang, multimodal results: the hash of
an input image is the key in the radix tree.  An image becomes a run of keys
from FNV-1a 64 of its bytes (Fowler, Noll, Vo) and the splitmix64 finaliser
(Steele, Lea, Flood 2014), all negative so no text token equals one.

Parity status: pinned by tests/test_oracle_pins.py -- the block cache against
the closed form of reuse vs shared-prefix length (16 * floor(L / 16) for
blocks, L for the radix tree, the comparison section 3 draws), the churn
counts and the cyclic sweep of section 6, and equality with the (separately
pinned) radix-tree oracle on block-aligned traces; image keys against the
published FNV-1a and splitmix64 test values.
"""
from __future__ import annotations

import bisect

OK, ERR_ARG, ERR_NOMEM, ERR_STATE = 0, -1, -2, -3
FREE, HELD, CACHED = 0, 1, 2
MASK64 = (1 << 64) - 1


class _Block:
    def __init__(self, bid, parent, tokens, slots, depth):
        self.id = bid
        self.parent = parent          # block id (None for the root)
        self.tokens = tuple(tokens)
        self.slots = list(slots)
        self.depth = depth
        self.ref = 0
        self.stamp = 0


class OracleBlockCache:
    """Same method names and return shapes as the product's BlockCache."""

    def __init__(self, pool_slots: int, block_tokens: int = 16):
        self.B = int(block_tokens)
        self.pool = int(pool_slots)
        self.state = [FREE] * self.pool
        self.free_list = list(range(self.pool))   # kept sorted
        self.blocks = {0: _Block(0, None, (), (), 0)}
        self.next_id = 1
        self.clock = 0
        self.st = dict(match_calls=0, match_tokens=0, match_hits=0, match_hit_tokens=0, insert_calls=0,
                       insert_new_tokens=0, insert_dup_freed=0, evicted_nodes=0, evicted_tokens=0)

    def uncached_tail(self, n: int) -> int:
        return int(n) % self.B

    # a child block of `parent` with these tokens, or None
    def _child(self, parent_id, tokens):
        for b in self.blocks.values():
            if b.parent == parent_id and b.tokens == tuple(tokens):
                return b
        return None

    def _chain(self, tok):
        """Blocks matched along tok from the root: [root, b1, b2, ...]."""
        chain = [self.blocks[0]]
        k = 0
        while (k + 1) * self.B <= len(tok):
            b = self._child(chain[-1].id, [int(x) for x in tok[k * self.B:(k + 1) * self.B]])
            if b is None:
                break
            chain.append(b)
            k += 1
        return chain

    def match(self, tokens, pin: bool):
        tok = [int(x) for x in tokens]
        chain = self._chain(tok)
        self.clock += 1
        for b in chain:
            b.stamp = self.clock
            if pin:
                b.ref += 1
        slots = [s for b in chain[1:] for s in b.slots]
        m = len(slots)
        self.st["match_calls"] += 1
        self.st["match_tokens"] += len(tok)
        self.st["match_hits"] += int(m > 0)
        self.st["match_hit_tokens"] += m
        return OK, m, _arr(slots), chain[-1].id

    def insert(self, tokens, slots, pin: bool):
        tok = [int(x) for x in tokens]
        sl = [int(x) for x in slots]
        n = len(tok)
        if any(s < 0 or s >= self.pool for s in sl):
            return ERR_ARG, 0, -1, _arr([])
        chain = self._chain(tok)
        have = [s for b in chain[1:] for s in b.slots]
        m = len(have)
        seen = set()
        for i in range(n):
            if i < m and sl[i] == have[i]:
                continue
            if self.state[sl[i]] != HELD or sl[i] in seen:
                return ERR_STATE, 0, -1, _arr([])
            seen.add(sl[i])
        self.clock += 1
        nb = n // self.B
        for j in range(len(chain) - 1, nb):
            blk = _Block(self.next_id, chain[-1].id, tok[j * self.B:(j + 1) * self.B],
                         sl[j * self.B:(j + 1) * self.B], chain[-1].depth + 1)
            self.next_id += 1
            self.blocks[blk.id] = blk
            for s in blk.slots:
                self.state[s] = CACHED
            chain.append(blk)
        dup = 0
        for i in range(m):
            if sl[i] != have[i]:
                self._give_back(sl[i])
                dup += 1
        for b in chain:
            b.stamp = self.clock
            if pin:
                b.ref += 1
        canon = [have[i] if i < m else sl[i] for i in range(n)]
        self.st["insert_calls"] += 1
        self.st["insert_new_tokens"] += (nb - (m // self.B)) * self.B
        self.st["insert_dup_freed"] += dup
        return OK, m, chain[-1].id, _arr(canon)

    def release(self, node: int):
        b = self.blocks.get(int(node))
        if b is None or b.ref <= 0:
            return ERR_STATE
        while b is not None:
            b.ref -= 1
            b = self.blocks[b.parent] if b.parent is not None else None
        return OK

    def evict(self, n_tokens: int, log_cap: int = 4096):
        if n_tokens < 0:
            return ERR_ARG, 0, _arr64([])
        freed, log = 0, []
        while freed < n_tokens:
            cands = [b for b in self.blocks.values() if b.id != 0 and b.ref == 0]
            if not cands:
                break
            v = min(cands, key=lambda b: (b.stamp, -b.depth, b.id))
            del self.blocks[v.id]
            for s in v.slots:
                self._give_back(s)
            freed += self.B
            log.append(v.id)
        self.st["evicted_nodes"] += len(log)
        self.st["evicted_tokens"] += freed
        return OK, freed, _arr64(log[:log_cap])

    def alloc(self, n: int):
        if n < 0:
            return ERR_ARG, _arr([])
        if n > len(self.free_list):
            return ERR_NOMEM, _arr([])
        out = self.free_list[:n]
        del self.free_list[:n]
        for s in out:
            self.state[s] = HELD
        return OK, _arr(out)

    def free(self, slots):
        sl = [int(x) for x in slots]
        if any(s < 0 or s >= self.pool for s in sl):
            return ERR_ARG
        if len(set(sl)) != len(sl) or any(self.state[s] != HELD for s in sl):
            return ERR_STATE
        for s in sl:
            self._give_back(s)
        return OK

    def sched_order(self, policy: int, prompts):
        if policy not in (0, 1):
            return ERR_ARG, _arr([])
        idx = list(range(len(prompts)))
        if policy == 1:
            lens = [(len(self._chain([int(x) for x in p])) - 1) * self.B for p in prompts]
            idx.sort(key=lambda i: (-lens[i], i))
        return OK, _arr(idx)

    def stats(self) -> dict:
        held = sum(1 for s in self.state if s == HELD)
        cached = sum(1 for s in self.state if s == CACHED)
        d = dict(pool=self.pool, free=len(self.free_list), caller=held, tree_tokens=cached,
                 nodes=len(self.blocks), pins=self.blocks[0].ref, clock=self.clock)
        d.update(self.st)
        return d

    def _give_back(self, s):
        self.state[s] = FREE
        bisect.insort(self.free_list, s)


class OracleBlockServer:
    """The scheduling round and the commits of a serving loop over this block
    cache, written out here as the radix oracle's oracle_admit and
    oracle_commit state them (note 49, sections 4 and 5): order the prompts;
    in that order match with a pin; a request that will decode starts at
    min(matched, prompt_len - 1), a prefill-only one at matched; take slots
    for the uncached part plus max_new, evicting the shortfall first when
    fewer are free; a request that still does not fit drops its pin and ends
    the round; max_batch (> 0) ends it too.  After prefill the prompt is
    inserted (pinned if the request will decode) and the admission pin
    dropped; at finish prompt + outputs are inserted unpinned and the pin
    dropped.  Only whole blocks enter the cache, so the slots of a request's
    partial last block go back to the pool when the request is done with
    them (after prefill for a prefill-only request, else at finish)."""

    def __init__(self, cache: OracleBlockCache):
        self.cache = cache

    def admit(self, pending: list, policy: int = 1, max_batch: int | None = None):
        c = self.cache
        st, order = c.sched_order(policy, [r.tokens[:r.prompt_len] for r in pending])
        assert st == OK
        admitted = []
        for i in order.tolist():
            if max_batch and len(admitted) >= max_batch:
                break
            r = pending[i]
            st, m, mslots, node = c.match(r.tokens[:r.prompt_len], True)
            assert st == OK
            first = min(m, r.prompt_len - 1) if r.max_new > 0 else m
            need = r.prompt_len - first + r.max_new
            if len(c.free_list) < need:
                c.evict(need - len(c.free_list))
            st, new = c.alloc(need)
            if st != OK:
                assert c.release(node) == OK
                break
            r.matched, r.first, r.node = m, first, node
            r.slots = _arr(list(mslots[:first]) + list(new))
            admitted.append(r)
        took = {id(r) for r in admitted}
        return admitted, [r for r in pending if id(r) not in took]

    def _done_with(self, r, n):
        k = n % self.cache.B
        if k:
            assert self.cache.free(r.slots[n - k:n]) == OK

    def commit_prompts(self, batch: list):
        for r in batch:
            L = r.prompt_len
            st, present, node, canon = self.cache.insert(r.tokens[:L], r.slots[:L], r.max_new > 0)
            assert st == OK
            r.slots[:L] = canon
            assert self.cache.release(r.node) == OK
            r.node = node if r.max_new > 0 else -1
            if r.max_new == 0:
                self._done_with(r, L)

    def finish(self, batch: list):
        for r in batch:
            if r.max_new == 0:
                continue
            n = r.prompt_len + r.max_new
            st, present, node, canon = self.cache.insert(r.tokens[:n], r.slots[:n], False)
            assert st == OK
            r.slots[:n] = canon
            assert self.cache.release(r.node) == OK
            r.node = -1
            self._done_with(r, n)


def _arr(x):
    import numpy as np
    return np.asarray(x, dtype=np.int32)


def _arr64(x):
    import numpy as np
    return np.asarray(x, dtype=np.int64)


# ------------------------------------------------------------------ image keys
def fnv1a64(data: bytes) -> int:
    """FNV-1a, 64 bits: offset basis 14695981039346656037, prime 1099511628211."""
    h = 14695981039346656037
    for byte in data:
        h ^= byte
        h = (h * 1099511628211) & MASK64
    return h


def splitmix64_finalise(z: int) -> int:
    """The output function of splitmix64 (Steele, Lea, Flood 2014)."""
    z &= MASK64
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & MASK64
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & MASK64
    return z ^ (z >> 31)


def image_key(data: bytes, n_tokens: int) -> list:
    """Key i = -1 - (top 30 bits of the finaliser of hash + (i+1) * golden gamma)."""
    h = fnv1a64(bytes(data))
    gamma = 0x9E3779B97F4A7C15
    return [-1 - (splitmix64_finalise(h + (i + 1) * gamma) >> 34) for i in range(n_tokens)]
