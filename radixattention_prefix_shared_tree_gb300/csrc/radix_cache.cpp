// Host half of the library: the radix tree over token ids, reference-count
// pinning, LRU leaf eviction, the slot allocator of the shared KV pool and the
// scheduling order.  Rules follow "RadixAttention, eviction and cache churn"
// (inference-notes note 49), sections 2, 4 and 5, and the RadixAttention
// paragraph and nine-step walkthrough of the unite.ai article on SGLang; the
// open points are read as documented in include/radixattn.h.
//
// Layout, chosen for O(match length) lookups and O(log n) eviction:
//  * nodes live in a flat vector and are recycled through a free list; a
//    node's token run and slot run are (offset, length) views into two
//    parallel append-only arenas, so splitting an edge copies nothing;
//  * one hash map keyed by (parent index, first token) holds every edge;
//  * evictable leaves (no children, no pins, not the root) sit in an ordered
//    set keyed by (last access, id), so the next victim is its first element;
//  * free slots are a two-level bitmap (slot_pool.h), so "the n smallest free
//    ids" is a scan of set bits from the lowest non-empty word.

#include "../../include/radixattn.h"
#include "slot_pool.h"

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <new>
#include <set>
#include <string>
#include <unordered_map>
#include <utility>
#include <vector>

namespace {

using rc_pool::CACHED;
using rc_pool::FREE;
using rc_pool::HELD;

struct Rec {
    int64_t id = -1;
    int32_t parent = -1;
    int32_t nchild = 0;
    int64_t off = 0;   // run start in the arenas
    int32_t len = 0;   // run length
    int64_t ref = 0;
    uint64_t stamp = 0;
    bool live = false;
    bool in_lru = false;
    uint64_t lru_stamp = 0;  // stamp under which it sits in the LRU set
};

// Length of the common prefix of a[0..n) and b[0..n).  The whole range is
// tried first with one memcmp (vectorised in the C library; a full match is
// the common case), then 256-element blocks, then one element at a time.
inline int64_t common_prefix(const int32_t* a, const int32_t* b, int64_t n) {
    if (n <= 0) return 0;
    if (std::memcmp(a, b, (size_t)n * sizeof(int32_t)) == 0) return n;
    int64_t k = 0;
    while (k + 256 <= n && std::memcmp(a + k, b + k, 256 * sizeof(int32_t)) == 0) k += 256;
    while (a[k] == b[k]) ++k;  // a difference exists below n
    return k;
}

inline uint64_t edge_key(int32_t parent, int32_t first_tok) {
    return ((uint64_t)(uint32_t)parent << 32) | (uint32_t)first_tok;
}

}  // namespace

struct rc_cache : rc_pool::SlotPool {
    std::vector<Rec> recs;
    std::vector<int32_t> spare;      // recycled node indices
    std::vector<int32_t> tok_arena, slot_arena;
    int64_t arena_live = 0;
    std::unordered_map<uint64_t, int32_t> edges;
    std::unordered_map<int64_t, int32_t> by_id;
    std::set<std::pair<uint64_t, int64_t>> lru;
    uint64_t clock = 0;
    int64_t next_id = 0;
    int64_t n_nodes = 0;

    std::vector<int32_t> path;       // scratch
    std::vector<int32_t> scratch_slots;

    int64_t match_calls = 0, match_tokens = 0, match_hits = 0, match_hit_tokens = 0;
    int64_t insert_calls = 0, insert_new_tokens = 0, insert_dup_freed = 0;
    int64_t evicted_nodes = 0, evicted_tokens = 0;

    // ------------------------------------------------------------- nodes
    int32_t new_rec(int32_t parent, int64_t off, int32_t len) {
        int32_t i;
        if (!spare.empty()) { i = spare.back(); spare.pop_back(); }
        else { i = (int32_t)recs.size(); recs.emplace_back(); }
        Rec& r = recs[(size_t)i];
        r = Rec();
        r.id = next_id++;
        r.parent = parent;
        r.off = off;
        r.len = len;
        r.live = true;
        by_id[r.id] = i;
        n_nodes += 1;
        return i;
    }
    const int32_t* toks(const Rec& r) const { return tok_arena.data() + r.off; }

    void lru_out(int32_t i) {
        Rec& r = recs[(size_t)i];
        if (r.in_lru) { lru.erase({r.lru_stamp, r.id}); r.in_lru = false; }
    }
    void lru_fix(int32_t i) {  // put node i in or out of the candidate set per its state
        Rec& r = recs[(size_t)i];
        bool want = i != 0 && r.nchild == 0 && r.ref == 0;
        if (r.in_lru && (!want || r.lru_stamp != r.stamp)) lru_out(i);
        if (want && !r.in_lru) { lru.insert({r.stamp, r.id}); r.in_lru = true; r.lru_stamp = r.stamp; }
    }

    // Split node i after k tokens; returns the new upper node.
    int32_t split(int32_t i, int32_t k) {
        Rec lower = recs[(size_t)i];
        int32_t up = new_rec(lower.parent, lower.off, k);  // may reallocate recs
        Rec& L = recs[(size_t)i];
        Rec& U = recs[(size_t)up];
        edges[edge_key(L.parent, tok_arena[(size_t)L.off])] = up;
        L.off += k;
        L.len -= k;
        L.parent = up;
        edges[edge_key(up, tok_arena[(size_t)L.off])] = i;
        U.nchild = 1;
        U.ref = L.ref;
        U.stamp = clock;
        return up;
    }

    // Descend along tok[0..n) without changing anything.  Returns the matched
    // length; `pth` (if given) receives root..the last node matched whole;
    // `sl` (if given, room for n) receives the matched slots.  A match that
    // stops inside an edge leaves that child in *mid and its matched count in
    // *mid_k (else *mid = -1).
    //
    // from / from_depth: start below node `from`, whose path from the root
    // spells tok[0..from_depth) (the caller knows it: a pinned node the same
    // tokens reached before); positions below from_depth are neither
    // compared nor copied to `sl`.  known >= 0: the match is known to be
    // exactly `known` tokens long (a walk of the same tokens since which no
    // node was removed), so tokens are not compared either.
    int64_t walk(const int32_t* tok, int64_t n, std::vector<int32_t>* pth, int32_t* sl, int32_t* mid,
                 int32_t* mid_k, int32_t from = 0, int64_t from_depth = 0, int64_t known = -1) const {
        int32_t cur = from;
        if (pth) {
            pth->clear();
            for (int32_t k = from; k >= 0; k = recs[(size_t)k].parent) pth->push_back(k);
            std::reverse(pth->begin(), pth->end());
        }
        if (mid) *mid = -1;
        int64_t i = from_depth;
        const int64_t end = known >= 0 ? known : n;
        while (i < end) {
            auto it = edges.find(edge_key(cur, tok[i]));
            if (it == edges.end()) break;
            int32_t c = it->second;
            const Rec& r = recs[(size_t)c];
            int64_t lim = std::min<int64_t>(r.len, end - i);
            int64_t k = known >= 0 ? lim : 1 + common_prefix(toks(r) + 1, tok + i + 1, lim - 1);
            if (sl) std::memcpy(sl + i, slot_arena.data() + r.off, (size_t)k * 4);
            i += k;
            if (k < r.len) {
                if (mid) { *mid = c; *mid_k = (int32_t)k; }
                break;
            }
            cur = c;
            if (pth) pth->push_back(cur);
        }
        return i;
    }

    // Tokens on the path root..node i (its depth).
    int64_t depth(int32_t i) const {
        int64_t d = 0;
        for (; i > 0; i = recs[(size_t)i].parent) d += recs[(size_t)i].len;
        return d;
    }

    // walk() with the end of the match made a node boundary: a stop inside
    // an edge splits it and the upper part ends `pth`.
    int64_t descend(const int32_t* tok, int64_t n, std::vector<int32_t>* pth, int32_t* sl, int64_t known = -1) {
        int32_t mid = -1, k = 0;
        int64_t m = walk(tok, n, pth, sl, &mid, &k, 0, 0, known);
        if (mid >= 0) {
            int32_t up = split(mid, k);
            if (pth) pth->push_back(up);
        }
        return m;
    }

    // Stamp the path with the clock (and pin it); one candidate-set update per node.
    void touch(const std::vector<int32_t>& pth, bool and_pin) {
        for (int32_t i : pth) {
            Rec& r = recs[(size_t)i];
            r.stamp = clock;
            if (and_pin) r.ref += 1;
            lru_fix(i);
        }
    }

    void maybe_compact() {
        int64_t sz = (int64_t)tok_arena.size();
        if (sz < (1 << 20) || sz < 3 * arena_live) return;
        std::vector<int32_t> nt, ns;
        nt.reserve((size_t)arena_live * 2);
        ns.reserve((size_t)arena_live * 2);
        for (Rec& r : recs) {
            if (!r.live) continue;
            int64_t o = (int64_t)nt.size();
            nt.insert(nt.end(), tok_arena.begin() + r.off, tok_arena.begin() + r.off + r.len);
            ns.insert(ns.end(), slot_arena.begin() + r.off, slot_arena.begin() + r.off + r.len);
            r.off = o;
        }
        tok_arena.swap(nt);
        slot_arena.swap(ns);
    }

    void dump_rec(int32_t i, const std::vector<std::vector<int32_t>>& kids, std::string& s) const {
        const Rec& r = recs[(size_t)i];
        char b[96];
        std::snprintf(b, sizeof b, "%lld %lld %lld %llu %d:", (long long)r.id,
                      (long long)(r.parent >= 0 ? recs[(size_t)r.parent].id : -1),
                      (long long)r.ref, (unsigned long long)r.stamp, r.len);
        s += b;
        for (int32_t k = 0; k < r.len; ++k) { s += ' '; s += std::to_string(tok_arena[(size_t)(r.off + k)]); }
        s += " |";
        for (int32_t k = 0; k < r.len; ++k) { s += ' '; s += std::to_string(slot_arena[(size_t)(r.off + k)]); }
        s += '\n';
        for (int32_t c : kids[(size_t)i]) dump_rec(c, kids, s);
    }
};

extern "C" {

rc_status rc_create(int64_t pool_slots, rc_cache** out) {
    if (!out || pool_slots < 0 || pool_slots > 0x7FFFFFFF) return RC_ERR_ARG;
    *out = nullptr;
    rc_cache* c = new (std::nothrow) rc_cache();
    if (!c) return RC_ERR_NOMEM;
    try {
        c->init_slots(pool_slots);
        c->new_rec(-1, 0, 0);  // root: index 0, id 0
    } catch (...) {
        delete c;
        return RC_ERR_NOMEM;
    }
    *out = c;
    return RC_OK;
}

void rc_destroy(rc_cache* c) { delete c; }

}  // extern "C"

namespace {

// rc_match_prefix; known >= 0: the match length is already known (see walk).
rc_status match_impl(rc_cache* c, const int32_t* tok, int64_t n, int pin, int64_t* matched, int32_t* out_slots,
                     rc_node* out_node, int64_t known) {
    if (!c || n < 0 || (n > 0 && !tok) || !matched || !out_node) return RC_ERR_ARG;
    c->clock += 1;
    int64_t m = c->descend(tok, n, &c->path, out_slots, known);
    c->touch(c->path, pin != 0);
    *matched = m;
    *out_node = c->recs[(size_t)c->path.back()].id;
    c->match_calls += 1;
    c->match_tokens += n;
    c->match_hit_tokens += m;
    c->match_hits += m > 0;
    return RC_OK;
}

}  // namespace

extern "C" {

rc_status rc_match_prefix(rc_cache* c, const int32_t* tok, int64_t n, int pin, int64_t* matched,
                          int32_t* out_slots, rc_node* out_node) {
    return match_impl(c, tok, n, pin, matched, out_slots, out_node, -1);
}

// Every slot id in [0, pool); a branch-free scan.
static bool slots_in_pool(const rc_cache* c, const int32_t* slots, int64_t n) {
    const uint32_t pool = (uint32_t)c->pool;  // at most 2^31 - 1: a negative id reads as >= pool
    uint32_t bad = 0;
    for (int64_t i = 0; i < n; ++i) bad |= (uint32_t)slots[i] >= pool;
    return bad == 0;
}

}  // extern "C"

namespace {

// rc_insert starting below node `from`, whose path spells tok[0..d0) and
// holds slots[0..d0) (see walk): those positions are neither compared nor
// range-checked again.  from = 0, d0 = 0 is rc_insert itself.
rc_status insert_impl(rc_cache* c, const int32_t* tok, const int32_t* slots, int64_t n, int pin,
                      int64_t* already_present, rc_node* out_node, int32_t* out_slots, int32_t from, int64_t d0) {
    if (!c || n < 0 || (n > 0 && (!tok || !slots)) || !already_present || !out_node) return RC_ERR_ARG;
    if (!slots_in_pool(c, slots + d0, n - d0)) return RC_ERR_ARG;
    std::vector<int32_t>& have = c->scratch_slots;
    if ((int64_t)have.size() < n) have.resize((size_t)n);
    int32_t mid = -1, mid_k = 0;
    int64_t m = c->walk(tok, n, &c->path, have.data(), &mid, &mid_k, from, d0);   // look first, change nothing
    c->new_epoch();
    // positions whose slot is already the cached one need no check
    const int64_t same = d0 + common_prefix(slots + d0, have.data() + d0, m - d0);
    for (int64_t i = same; i < n; ++i) {
        int32_t s = slots[i];
        if (i < m && s == have[(size_t)i]) continue;
        if (c->owner[(size_t)s] != HELD || c->mark[(size_t)s] == c->epoch) return RC_ERR_STATE;
        c->mark[(size_t)s] = c->epoch;
    }
    c->clock += 1;
    if (mid >= 0) c->path.push_back(c->split(mid, mid_k));   // the walk's end made a node boundary
    if (m < n) {
        int32_t parent = c->path.back();
        int64_t off = (int64_t)c->tok_arena.size();
        c->tok_arena.insert(c->tok_arena.end(), tok + m, tok + n);
        c->slot_arena.insert(c->slot_arena.end(), slots + m, slots + n);
        int32_t leaf = c->new_rec(parent, off, (int32_t)(n - m));
        c->edges[edge_key(parent, tok[m])] = leaf;
        c->recs[(size_t)parent].nchild += 1;
        c->lru_fix(parent);
        for (int64_t i = m; i < n; ++i) c->owner[(size_t)slots[i]] = CACHED;
        c->n_held -= n - m;
        c->n_cached += n - m;
        c->arena_live += n - m;
        c->path.push_back(leaf);
    }
    int64_t dup = 0;
    for (int64_t i = same; i < m; ++i) {
        int32_t s = slots[i];
        if (s == have[(size_t)i]) continue;
        c->owner[(size_t)s] = FREE;
        c->slot_set_free(s);
        dup += 1;
    }
    c->n_held -= dup;
    c->n_free += dup;
    c->touch(c->path, pin != 0);
    if (out_slots) {
        if (d0 && out_slots != slots) std::memmove(out_slots, slots, (size_t)d0 * 4);   // the tree's, by contract
        if (m > d0) std::memcpy(out_slots + d0, have.data() + d0, (size_t)(m - d0) * 4);
        if (n > m && out_slots != slots) std::memmove(out_slots + m, slots + m, (size_t)(n - m) * 4);
    }
    *already_present = m;
    *out_node = c->recs[(size_t)c->path.back()].id;
    c->insert_calls += 1;
    c->insert_new_tokens += n - m;
    c->insert_dup_freed += dup;
    return RC_OK;
}

}  // namespace

extern "C" {

rc_status rc_insert(rc_cache* c, const int32_t* tok, const int32_t* slots, int64_t n, int pin,
                    int64_t* already_present, rc_node* out_node, int32_t* out_slots) {
    return insert_impl(c, tok, slots, n, pin, already_present, out_node, out_slots, 0, 0);
}

rc_status rc_release(rc_cache* c, rc_node node) {
    if (!c) return RC_ERR_ARG;
    auto it = c->by_id.find(node);
    if (it == c->by_id.end()) return RC_ERR_STATE;
    int32_t i = it->second;
    if (c->recs[(size_t)i].ref <= 0) return RC_ERR_STATE;
    for (; i >= 0; i = c->recs[(size_t)i].parent) {
        c->recs[(size_t)i].ref -= 1;
        c->lru_fix(i);
    }
    return RC_OK;
}

rc_status rc_evict(rc_cache* c, int64_t n_tokens, int64_t* freed, int64_t* log, int64_t log_cap,
                   int64_t* n_evicted) {
    if (!c || n_tokens < 0 || !freed || !n_evicted || (log_cap > 0 && !log)) return RC_ERR_ARG;
    int64_t got = 0, cnt = 0;
    while (got < n_tokens && !c->lru.empty()) {
        int64_t id = c->lru.begin()->second;
        c->lru.erase(c->lru.begin());
        int32_t i = c->by_id[id];
        Rec& r = c->recs[(size_t)i];
        r.in_lru = false;
        for (int32_t k = 0; k < r.len; ++k) {
            int32_t s = c->slot_arena[(size_t)(r.off + k)];
            c->owner[(size_t)s] = FREE;
            c->slot_set_free(s);
        }
        c->n_free += r.len;
        c->n_cached -= r.len;
        c->arena_live -= r.len;
        got += r.len;
        c->edges.erase(edge_key(r.parent, c->tok_arena[(size_t)r.off]));
        int32_t p = r.parent;
        c->recs[(size_t)p].nchild -= 1;
        if (log && cnt < log_cap) log[cnt] = id;
        cnt += 1;
        c->evicted_nodes += 1;
        c->evicted_tokens += r.len;
        r.live = false;
        c->by_id.erase(id);
        c->n_nodes -= 1;
        c->spare.push_back(i);
        c->lru_fix(p);
    }
    c->maybe_compact();
    *freed = got;
    *n_evicted = cnt;
    return RC_OK;
}

rc_status rc_alloc(rc_cache* c, int64_t n, int32_t* out) {
    if (!c || n < 0 || (n > 0 && !out)) return RC_ERR_ARG;
    if (n > c->n_free) return RC_ERR_NOMEM;
    if (n) c->take_lowest(n, out);
    return RC_OK;
}

rc_status rc_free(rc_cache* c, const int32_t* slots, int64_t n) {
    if (!c || n < 0 || (n > 0 && !slots)) return RC_ERR_ARG;
    const int r = c->free_held(slots, n);
    return r == -1 ? RC_ERR_ARG : r == -2 ? RC_ERR_STATE : RC_OK;
}

}  // extern "C"

namespace {

// sched_order; peek (optional, room for n) receives each prompt's peek match
// length under RC_LPM (left untouched under RC_FCFS).
rc_status order_impl(rc_cache* c, int policy, const int32_t* const* prompts, const int64_t* lens, int32_t n,
                     int32_t* out_order, int64_t* peek) {
    if (!c || n < 0 || (n > 0 && (!prompts || !lens || !out_order))) return RC_ERR_ARG;
    if (policy != RC_FCFS && policy != RC_LPM) return RC_ERR_ARG;
    for (int32_t i = 0; i < n; ++i)
        if (lens[i] < 0 || (lens[i] > 0 && !prompts[i])) return RC_ERR_ARG;
    for (int32_t i = 0; i < n; ++i) out_order[i] = i;
    if (policy == RC_LPM && (n > 1 || peek)) {
        std::vector<std::pair<int64_t, int32_t>> key((size_t)n);
        for (int32_t i = 0; i < n; ++i) {
            const int64_t m = c->walk(prompts[i], lens[i], nullptr, nullptr, nullptr, nullptr);
            if (peek) peek[i] = m;
            key[(size_t)i] = {-m, i};
        }
        std::sort(key.begin(), key.end());  // (-match, index): longest first, then arrival
        for (int32_t i = 0; i < n; ++i) out_order[i] = key[(size_t)i].second;
    }
    return RC_OK;
}

}  // namespace

extern "C" {

rc_status sched_order(rc_cache* c, int policy, const int32_t* const* prompts, const int64_t* lens,
                      int32_t n, int32_t* out_order) {
    return order_impl(c, policy, prompts, lens, n, out_order, nullptr);
}

rc_status rc_admit(rc_cache* c, int policy, rc_request* reqs, int32_t n, int32_t max_batch, int32_t* out_order,
                   int32_t* n_admitted) {
    if (!c || n < 0 || (n > 0 && (!reqs || !out_order)) || !n_admitted) return RC_ERR_ARG;
    *n_admitted = 0;
    if (n == 0) return RC_OK;
    std::vector<const int32_t*> prompts((size_t)n);
    std::vector<int64_t> lens((size_t)n);
    for (int32_t i = 0; i < n; ++i) {
        const rc_request& r = reqs[i];
        if (r.prompt_len < 0 || r.max_new < 0 || (r.prompt_len > 0 && !r.tokens) || !r.slots ||
            (r.max_new > 0 && r.prompt_len == 0))
            return RC_ERR_ARG;
        prompts[(size_t)i] = r.tokens;
        lens[(size_t)i] = r.prompt_len;
        reqs[i].admitted = 0;
        reqs[i].node = -1;
    }
    std::vector<int32_t> order((size_t)n);
    std::vector<int64_t> peek((size_t)n, -1);
    rc_status st = order_impl(c, policy, prompts.data(), lens.data(), n, order.data(), peek.data());
    if (st != RC_OK) return st;
    // the LPM peeks stay exact match lengths until a node is removed: the
    // matches below only split edges (same tokens), pin and stamp
    const int64_t evicted0 = c->evicted_nodes;
    int32_t count = 0;
    for (int32_t k = 0; k < n; ++k) {
        if (max_batch > 0 && count >= max_batch) break;
        rc_request& r = reqs[order[(size_t)k]];
        int64_t m = 0;
        rc_node node = 0;
        const int64_t known = c->evicted_nodes == evicted0 ? peek[(size_t)order[(size_t)k]] : -1;
        // the matched slots land in the row itself (room for prompt_len + max_new >= matched);
        // the new ones then overwrite it from `first` on
        st = match_impl(c, r.tokens, r.prompt_len, 1, &m, r.slots, &node, known);
        if (st != RC_OK) return st;
        const int64_t first = r.max_new > 0 ? std::min(m, r.prompt_len - 1) : m;
        const int64_t need = r.prompt_len - first + r.max_new;
        int32_t* dst = r.slots + first;
        st = rc_alloc(c, need, dst);
        if (st == RC_ERR_NOMEM) {
            int64_t freed = 0, cnt = 0;
            st = rc_evict(c, need - c->n_free, &freed, nullptr, 0, &cnt);
            if (st != RC_OK) return st;
            st = rc_alloc(c, need, dst);
        }
        if (st != RC_OK) {
            if (st != RC_ERR_NOMEM) return st;
            rc_status rs = rc_release(c, node);
            if (rs != RC_OK) return rs;
            break;  // the first request that does not fit stops the round
        }
        r.matched = m;
        r.first = first;
        r.node = node;
        r.admitted = 1;
        out_order[count++] = order[(size_t)k];
    }
    *n_admitted = count;
    return RC_OK;
}

rc_status rc_commit(rc_cache* c, rc_request* reqs, const int32_t* idx, int32_t n, int mode) {
    if (!c || n < 0 || (n > 0 && (!reqs || !idx)) || (mode != RC_COMMIT_PREFILL && mode != RC_COMMIT_FINISH))
        return RC_ERR_ARG;
    for (int32_t k = 0; k < n; ++k) {
        rc_request& r = reqs[idx[k]];
        if (mode == RC_COMMIT_FINISH && r.max_new == 0) continue;
        const int64_t len = mode == RC_COMMIT_PREFILL ? r.prompt_len : r.prompt_len + r.max_new;
        const int pin = mode == RC_COMMIT_PREFILL && r.max_new > 0;
        // The request's pinned node spells its first tokens: the match of
        // rc_admit (slots[0..first) are its slots), or the prompt inserted
        // by the prefill commit (slots[0..prompt_len) are the tree's).  The
        // insert starts at its deepest ancestor within those positions.
        int32_t from = 0;
        int64_t d0 = 0;
        const auto it = c->by_id.find(r.node);
        if (it != c->by_id.end()) {
            const int64_t known = mode == RC_COMMIT_PREFILL ? r.first : r.prompt_len;
            int32_t k = it->second;
            int64_t d = c->depth(k);
            while (k > 0 && d > known) {
                d -= c->recs[(size_t)k].len;
                k = c->recs[(size_t)k].parent;
            }
            if (d <= known && known <= len) {
                from = k;
                d0 = d;
            }
        }
        int64_t present = 0;
        rc_node node = -1;
        rc_status st = insert_impl(c, r.tokens, r.slots, len, pin, &present, &node, r.slots, from, d0);
        if (st != RC_OK) return st;
        st = rc_release(c, r.node);
        if (st != RC_OK) return st;
        r.node = pin ? node : -1;
    }
    return RC_OK;
}

rc_status rc_cascade_plan(rc_cache* c, const rc_node* nodes, int32_t n, int32_t* seg_slots, int64_t seg_slots_cap,
                          int32_t* seg_indptr, int32_t* seg_row_indptr, int32_t* seg_rows, int32_t* req_seg_indptr,
                          int32_t* req_seg_pos, int64_t rows_cap, int64_t* private_start, int32_t seg_cap,
                          int32_t* n_seg, int64_t* n_seg_slots, int32_t* total_rows, int32_t* max_seg_len,
                          int32_t* max_seg_rows) {
    if (!c || n < 0 || (n > 0 && !nodes) || !seg_indptr || !seg_row_indptr || !req_seg_indptr || !private_start ||
        !n_seg || !n_seg_slots || !total_rows || !max_seg_len || !max_seg_rows || seg_cap < 0)
        return RC_ERR_ARG;
    // paths root..node (root excluded), as record indices
    std::vector<std::vector<int32_t>> paths((size_t)n);
    std::unordered_map<int32_t, int32_t> uses;
    for (int32_t i = 0; i < n; ++i) {
        auto it = c->by_id.find(nodes[i]);
        if (it == c->by_id.end()) return RC_ERR_STATE;
        for (int32_t k = it->second; k > 0; k = c->recs[(size_t)k].parent) paths[(size_t)i].push_back(k);
        std::reverse(paths[(size_t)i].begin(), paths[(size_t)i].end());
        for (int32_t k : paths[(size_t)i]) uses[k] += 1;
    }
    // segments in order of first appearance along the requests' paths
    std::unordered_map<int32_t, int32_t> seg_of;
    std::vector<int32_t> seg_rec;
    for (int32_t i = 0; i < n; ++i)
        for (int32_t k : paths[(size_t)i]) {
            if (uses[k] < 2) break;
            if (seg_of.emplace(k, (int32_t)seg_rec.size()).second) seg_rec.push_back(k);
        }
    const int32_t ns = (int32_t)seg_rec.size();
    if (ns > seg_cap) return RC_ERR_NOMEM;
    std::vector<std::vector<int32_t>> rows_of((size_t)ns);
    req_seg_indptr[0] = 0;
    int64_t pos_total = 0;
    for (int32_t i = 0; i < n; ++i) {
        int64_t priv = 0;
        for (int32_t k : paths[(size_t)i]) {
            if (uses[k] < 2) break;
            rows_of[(size_t)seg_of[k]].push_back(i);
            priv += c->recs[(size_t)k].len;
            pos_total += 1;
        }
        private_start[i] = priv;
    }
    if (pos_total > rows_cap || (pos_total > 0 && (!seg_rows || !req_seg_pos))) return RC_ERR_NOMEM;
    int64_t nslots = 0;
    int32_t mlen = 0, mrows = 0, rpos = 0;
    seg_indptr[0] = 0;
    seg_row_indptr[0] = 0;
    std::vector<std::vector<int32_t>> pos_of((size_t)n);
    for (int32_t s = 0; s < ns; ++s) {
        const Rec& r = c->recs[(size_t)seg_rec[(size_t)s]];
        if (nslots + r.len > seg_slots_cap || !seg_slots) return RC_ERR_NOMEM;
        std::memcpy(seg_slots + nslots, c->slot_arena.data() + r.off, (size_t)r.len * 4);
        nslots += r.len;
        seg_indptr[s + 1] = (int32_t)nslots;
        mlen = std::max(mlen, r.len);
        const auto& rw = rows_of[(size_t)s];
        mrows = std::max(mrows, (int32_t)rw.size());
        for (int32_t b : rw) {
            pos_of[(size_t)b].push_back(rpos);
            seg_rows[rpos++] = b;
        }
        seg_row_indptr[s + 1] = rpos;
    }
    int32_t q = 0;
    for (int32_t i = 0; i < n; ++i) {
        for (int32_t p2 : pos_of[(size_t)i]) req_seg_pos[q++] = p2;
        req_seg_indptr[i + 1] = q;
    }
    *n_seg = ns;
    *n_seg_slots = nslots;
    *total_rows = rpos;
    *max_seg_len = mlen;
    *max_seg_rows = mrows;
    return RC_OK;
}

rc_status rc_stats(rc_cache* c, rc_stats_t* o) {
    if (!c || !o) return RC_ERR_ARG;
    o->pool_slots = c->pool;
    o->free_slots = c->n_free;
    o->caller_slots = c->n_held;
    o->tree_tokens = c->n_cached;
    o->nodes = c->n_nodes;
    o->match_calls = c->match_calls;
    o->match_tokens = c->match_tokens;
    o->match_hits = c->match_hits;
    o->match_hit_tokens = c->match_hit_tokens;
    o->insert_calls = c->insert_calls;
    o->insert_new_tokens = c->insert_new_tokens;
    o->insert_dup_freed = c->insert_dup_freed;
    o->evicted_nodes = c->evicted_nodes;
    o->evicted_tokens = c->evicted_tokens;
    o->pins = c->recs[0].ref;
    o->clock = (int64_t)c->clock;
    return RC_OK;
}

rc_status rc_dump(rc_cache* c, char* buf, int64_t cap, int64_t* needed) {
    if (!c || !needed || cap < 0 || (cap > 0 && !buf)) return RC_ERR_ARG;
    std::vector<std::vector<int32_t>> kids(c->recs.size());
    for (size_t i = 1; i < c->recs.size(); ++i)
        if (c->recs[i].live) kids[(size_t)c->recs[i].parent].push_back((int32_t)i);
    for (auto& k : kids)
        std::sort(k.begin(), k.end(), [&](int32_t a, int32_t b) {
            return c->tok_arena[(size_t)c->recs[(size_t)a].off] < c->tok_arena[(size_t)c->recs[(size_t)b].off];
        });
    std::string s;
    c->dump_rec(0, kids, s);
    *needed = (int64_t)s.size();
    if (cap > 0) {
        int64_t k = std::min<int64_t>(cap - 1, (int64_t)s.size());
        std::memcpy(buf, s.data(), (size_t)k);
        buf[k] = 0;
    }
    return RC_OK;
}

}  // extern "C"

// ------------------------------------------------------------------ image keys
// The unite.ai article on SGLang, multimodal results: for RadixAttention the
// hash of an input image is computed and used as the key in the tree, so the
// KV of the image's tokens is reused whenever the same image comes again.
// Here an image becomes a run of n_tokens keys (the model's image-token
// count), all derived from a hash of its bytes and all negative, so they
// never equal a text token id (>= 0).  Byte hash: FNV-1a 64 (Fowler, Noll,
// Vo); key i: the top 30 bits of the splitmix64 finaliser (Steele, Lea,
// Flood 2014) of hash + (i+1) * 0x9E3779B97F4A7C15, as -1 - bits.
namespace {
inline uint64_t image_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
}  // namespace

extern "C" rc_status rc_image_key(const void* data, int64_t bytes, int32_t n_tokens, int32_t* out) {
    if (bytes < 0 || n_tokens < 0 || (bytes > 0 && !data) || (n_tokens > 0 && !out)) return RC_ERR_ARG;
    const unsigned char* p = static_cast<const unsigned char*>(data);
    uint64_t h = 0xCBF29CE484222325ull;
    for (int64_t i = 0; i < bytes; ++i) {
        h ^= p[i];
        h *= 0x100000001B3ull;
    }
    for (int32_t i = 0; i < n_tokens; ++i)
        out[i] = -1 - (int32_t)(image_mix(h + (uint64_t)(i + 1) * 0x9E3779B97F4A7C15ull) >> 34);
    return RC_OK;
}
