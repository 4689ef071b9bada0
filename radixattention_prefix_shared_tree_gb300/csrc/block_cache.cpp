// Host comparator: a prefix cache over fixed-size token blocks, the scheme
// "RadixAttention, eviction and cache churn" (inference-notes note 49),
// section 3, sets against the radix tree: each block of B = 16 tokens is
// keyed by a hash chain over everything before it, a lookup matches whole
// blocks only, blocks are shared by reference count and the least recently
// used go first.  It draws on the same slot pool (slot_pool.h), has the same
// call shapes and the same LRU clock as the radix tree, so on one trace the
// two differ only in the granularity of the match.
//
// Readings where the section gives a table rather than rules:
//  * only a full block is cached: tokens [B*i, B*i+B) of a sequence, known by
//    the block before it and its own B tokens (a hash chain without
//    collisions: the key is compared exactly, the hash only indexes);
//  * a lookup walks whole blocks from the start and stops at the first block
//    that is not cached, so a match is a multiple of B long;
//  * insert caches every full block not cached yet; the partial last block
//    stays with the caller (held slots), who frees it once the request no
//    longer needs it;
//  * each match and each insert advance the LRU clock by one and stamp every
//    block of the touched chain (the root, i.e. the empty chain, included);
//    a pin counts on every block of the chain;
//  * eviction takes any block without pins (never the root), least recently
//    used first; blocks stamped by one call lie on one chain, and of those the
//    one farthest from the start goes first, so a chain shrinks from its end;
//    it stops as soon as the freed count reaches the request.
//
// Layout: blocks in a flat vector recycled through a free list, their tokens
// and slots in two arrays of B entries per block index, a hash index from
// (parent id, tokens) to block, and the candidates in an ordered set keyed by
// (last access, -depth, id).

#include "../../include/radixattn.h"
#include "slot_pool.h"

#include <algorithm>
#include <cstring>
#include <new>
#include <set>
#include <tuple>
#include <unordered_map>
#include <vector>

namespace {

using rc_pool::CACHED;
using rc_pool::HELD;

struct Blk {
    int64_t id = -1;
    int32_t parent = -1;
    int32_t depth = 0;     // blocks on the chain up to and including this one
    int64_t ref = 0;
    uint64_t stamp = 0;
    uint64_t key = 0;      // index hash of (parent id, tokens)
    bool live = false;
    bool in_lru = false;
    uint64_t lru_stamp = 0;
};

using LruKey = std::tuple<uint64_t, int32_t, int64_t>;  // (last access, -depth, id)

uint64_t block_key(int64_t parent_id, const int32_t* t, int32_t B) {
    uint64_t h = 0x9E3779B97F4A7C15ull ^ ((uint64_t)parent_id * 0xBF58476D1CE4E5B9ull);
    for (int32_t i = 0; i < B; ++i) {
        h ^= (uint32_t)t[i];
        h *= 0x100000001B3ull;
        h ^= h >> 29;
    }
    return h;
}

}  // namespace

struct bc_cache : rc_pool::SlotPool {
    int32_t B = 16;
    std::vector<Blk> blks;
    std::vector<int32_t> spare;
    std::vector<int32_t> btok, bslot;   // B entries per block index
    std::unordered_multimap<uint64_t, int32_t> index;
    std::unordered_map<int64_t, int32_t> by_id;
    std::set<LruKey> lru;
    uint64_t clock = 0;
    int64_t next_id = 0;
    int64_t n_blocks = 0;
    std::vector<int32_t> path;
    std::vector<int32_t> have;

    int64_t match_calls = 0, match_tokens = 0, match_hits = 0, match_hit_tokens = 0;
    int64_t insert_calls = 0, insert_new_tokens = 0, insert_dup_freed = 0;
    int64_t evicted_blocks = 0, evicted_tokens = 0;

    int32_t lookup(int32_t parent, const int32_t* t) const {
        auto r = index.equal_range(block_key(blks[(size_t)parent].id, t, B));
        for (auto it = r.first; it != r.second; ++it) {
            const int32_t i = it->second;
            if (blks[(size_t)i].parent == parent &&
                std::memcmp(btok.data() + (size_t)i * B, t, (size_t)B * sizeof(int32_t)) == 0)
                return i;
        }
        return -1;
    }
    int32_t new_blk(int32_t parent, const int32_t* t, const int32_t* s) {
        int32_t i;
        if (!spare.empty()) {
            i = spare.back();
            spare.pop_back();
        } else {
            i = (int32_t)blks.size();
            blks.emplace_back();
            btok.resize(btok.size() + (size_t)B);
            bslot.resize(bslot.size() + (size_t)B);
        }
        Blk& b = blks[(size_t)i];
        b = Blk();
        b.id = next_id++;
        b.parent = parent;
        b.depth = parent >= 0 ? blks[(size_t)parent].depth + 1 : 0;
        b.live = true;
        if (parent >= 0) {
            std::memcpy(btok.data() + (size_t)i * B, t, (size_t)B * sizeof(int32_t));
            std::memcpy(bslot.data() + (size_t)i * B, s, (size_t)B * sizeof(int32_t));
            b.key = block_key(blks[(size_t)parent].id, t, B);
            index.emplace(b.key, i);
        }
        by_id[b.id] = i;
        n_blocks += 1;
        return i;
    }
    void lru_fix(int32_t i) {
        Blk& b = blks[(size_t)i];
        const bool eligible = i != 0 && b.live && b.ref == 0;
        if (b.in_lru && (!eligible || b.lru_stamp != b.stamp)) {
            lru.erase(LruKey{b.lru_stamp, -b.depth, b.id});
            b.in_lru = false;
        }
        if (eligible && !b.in_lru) {
            lru.insert(LruKey{b.stamp, -b.depth, b.id});
            b.in_lru = true;
            b.lru_stamp = b.stamp;
        }
    }
    // Whole cached blocks along tok[0..n): path receives root..last block,
    // `sl` (if given) their slots.  Returns the number of blocks.
    int64_t descend(const int32_t* tok, int64_t n, std::vector<int32_t>& pth, std::vector<int32_t>* sl) const {
        pth.clear();
        pth.push_back(0);
        int32_t cur = 0;
        int64_t k = 0;
        while ((k + 1) * B <= n) {
            const int32_t i = lookup(cur, tok + k * B);
            if (i < 0) break;
            pth.push_back(i);
            if (sl) sl->insert(sl->end(), bslot.begin() + (size_t)i * B, bslot.begin() + (size_t)(i + 1) * B);
            cur = i;
            ++k;
        }
        return k;
    }
    void touch_and_pin(bool pin) {
        for (int32_t i : path) {
            blks[(size_t)i].stamp = clock;
            if (pin) blks[(size_t)i].ref += 1;
            lru_fix(i);
        }
    }
    void remove_blk(int32_t i) {
        Blk& b = blks[(size_t)i];
        if (b.in_lru) lru.erase(LruKey{b.lru_stamp, -b.depth, b.id});
        auto r = index.equal_range(b.key);
        for (auto it = r.first; it != r.second; ++it)
            if (it->second == i) {
                index.erase(it);
                break;
            }
        by_id.erase(b.id);
        for (int32_t j = 0; j < B; ++j) release_slot(bslot[(size_t)i * B + j]);
        b = Blk();
        spare.push_back(i);
        n_blocks -= 1;
    }
};

extern "C" {

rc_status bc_create(int64_t pool_slots, int32_t block_tokens, bc_cache** out) {
    if (!out || pool_slots < 0 || pool_slots > 0x7FFFFFFF || block_tokens < 1 || block_tokens > 4096)
        return RC_ERR_ARG;
    *out = nullptr;
    bc_cache* c = new (std::nothrow) bc_cache();
    if (!c) return RC_ERR_NOMEM;
    try {
        c->B = block_tokens;
        c->init_slots(pool_slots);
        c->new_blk(-1, nullptr, nullptr);  // root: index 0, id 0, the empty chain
    } catch (...) {
        delete c;
        return RC_ERR_NOMEM;
    }
    *out = c;
    return RC_OK;
}

void bc_destroy(bc_cache* c) { delete c; }

rc_status bc_match_prefix(bc_cache* c, const int32_t* tok, int64_t n, int pin, int64_t* matched,
                          int32_t* out_slots, rc_node* out_node) {
    if (!c || n < 0 || (n > 0 && !tok) || !matched || !out_node) return RC_ERR_ARG;
    try {
        c->have.clear();
        const int64_t k = c->descend(tok, n, c->path, out_slots ? &c->have : nullptr);
        c->clock += 1;
        c->touch_and_pin(pin != 0);
        const int64_t m = k * c->B;
        if (out_slots && m) std::memcpy(out_slots, c->have.data(), (size_t)m * sizeof(int32_t));
        *matched = m;
        *out_node = c->blks[(size_t)c->path.back()].id;
        c->match_calls += 1;
        c->match_tokens += n;
        c->match_hits += m > 0;
        c->match_hit_tokens += m;
    } catch (...) {
        return RC_ERR_NOMEM;
    }
    return RC_OK;
}

rc_status bc_insert(bc_cache* c, const int32_t* tok, const int32_t* slots, int64_t n, int pin,
                    int64_t* already_present, rc_node* out_node, int32_t* out_slots) {
    if (!c || n < 0 || (n > 0 && (!tok || !slots)) || !already_present || !out_node) return RC_ERR_ARG;
    for (int64_t i = 0; i < n; ++i)
        if (slots[i] < 0 || slots[i] >= c->pool) return RC_ERR_ARG;
    try {
        c->have.clear();
        const int64_t k = c->descend(tok, n, c->path, &c->have);
        const int64_t m = k * c->B;
        // every caller slot that is not the cached one must be held, once
        const uint32_t e = c->new_epoch();
        for (int64_t i = 0; i < n; ++i) {
            const int32_t s = slots[i];
            if (i < m && s == c->have[(size_t)i]) continue;
            if (c->owner[(size_t)s] != HELD || c->mark[(size_t)s] == e) return RC_ERR_STATE;
            c->mark[(size_t)s] = e;
        }
        c->clock += 1;
        const int64_t nb = n / c->B;
        int32_t cur = c->path.back();
        for (int64_t j = k; j < nb; ++j) {
            const int32_t i = c->new_blk(cur, tok + j * c->B, slots + j * c->B);
            for (int32_t q = 0; q < c->B; ++q) c->cache_slot(slots[j * c->B + q]);
            c->path.push_back(i);
            cur = i;
        }
        int64_t dup = 0;
        for (int64_t i = 0; i < m; ++i)
            if (slots[i] != c->have[(size_t)i]) {
                c->release_slot(slots[i]);
                dup += 1;
            }
        c->touch_and_pin(pin != 0);
        if (out_slots)
            for (int64_t i = 0; i < n; ++i) out_slots[i] = i < m ? c->have[(size_t)i] : slots[i];
        *already_present = m;
        *out_node = c->blks[(size_t)c->path.back()].id;
        c->insert_calls += 1;
        c->insert_new_tokens += (nb - k) * c->B;
        c->insert_dup_freed += dup;
    } catch (...) {
        return RC_ERR_NOMEM;
    }
    return RC_OK;
}

rc_status bc_release(bc_cache* c, rc_node node) {
    if (!c) return RC_ERR_ARG;
    auto it = c->by_id.find(node);
    if (it == c->by_id.end()) return RC_ERR_STATE;
    int32_t i = it->second;
    if (c->blks[(size_t)i].ref <= 0) return RC_ERR_STATE;
    for (; i >= 0; i = c->blks[(size_t)i].parent) {
        c->blks[(size_t)i].ref -= 1;
        c->lru_fix(i);
    }
    return RC_OK;
}

rc_status bc_evict(bc_cache* c, int64_t n_tokens, int64_t* freed, int64_t* log, int64_t log_cap,
                   int64_t* n_evicted) {
    if (!c || n_tokens < 0 || !freed || !n_evicted || log_cap < 0 || (log_cap > 0 && !log)) return RC_ERR_ARG;
    int64_t got = 0, cnt = 0;
    while (got < n_tokens && !c->lru.empty()) {
        const int64_t id = std::get<2>(*c->lru.begin());
        const int32_t i = c->by_id.at(id);
        c->remove_blk(i);
        if (cnt < log_cap) log[cnt] = id;
        cnt += 1;
        got += c->B;
    }
    c->evicted_blocks += cnt;
    c->evicted_tokens += got;
    *freed = got;
    *n_evicted = cnt;
    return RC_OK;
}

rc_status bc_alloc(bc_cache* c, int64_t n, int32_t* out) {
    if (!c || n < 0 || (n > 0 && !out)) return RC_ERR_ARG;
    if (n > c->n_free) return RC_ERR_NOMEM;
    if (n) c->take_lowest(n, out);
    return RC_OK;
}

rc_status bc_free(bc_cache* c, const int32_t* slots, int64_t n) {
    if (!c || n < 0 || (n > 0 && !slots)) return RC_ERR_ARG;
    const int r = c->free_held(slots, n);
    return r == -1 ? RC_ERR_ARG : r == -2 ? RC_ERR_STATE : RC_OK;
}

rc_status bc_sched_order(bc_cache* c, int policy, const int32_t* const* prompts, const int64_t* lens,
                         int32_t n, int32_t* out_order) {
    if (!c || n < 0 || (n > 0 && (!prompts || !lens || !out_order))) return RC_ERR_ARG;
    if (policy != RC_FCFS && policy != RC_LPM) return RC_ERR_ARG;
    for (int32_t i = 0; i < n; ++i)
        if (lens[i] < 0 || (lens[i] > 0 && !prompts[i])) return RC_ERR_ARG;
    for (int32_t i = 0; i < n; ++i) out_order[i] = i;
    if (policy == RC_FCFS) return RC_OK;
    try {
        std::vector<int64_t> len((size_t)n);
        std::vector<int32_t> pth;
        for (int32_t i = 0; i < n; ++i) len[(size_t)i] = c->descend(prompts[i], lens[i], pth, nullptr) * c->B;
        std::stable_sort(out_order, out_order + n,
                         [&](int32_t a, int32_t b) { return len[(size_t)a] > len[(size_t)b]; });
    } catch (...) {
        return RC_ERR_NOMEM;
    }
    return RC_OK;
}

rc_status bc_stats(bc_cache* c, rc_stats_t* o) {
    if (!c || !o) return RC_ERR_ARG;
    o->pool_slots = c->pool;
    o->free_slots = c->n_free;
    o->caller_slots = c->n_held;
    o->tree_tokens = c->n_cached;
    o->nodes = c->n_blocks;
    o->match_calls = c->match_calls;
    o->match_tokens = c->match_tokens;
    o->match_hits = c->match_hits;
    o->match_hit_tokens = c->match_hit_tokens;
    o->insert_calls = c->insert_calls;
    o->insert_new_tokens = c->insert_new_tokens;
    o->insert_dup_freed = c->insert_dup_freed;
    o->evicted_nodes = c->evicted_blocks;
    o->evicted_tokens = c->evicted_tokens;
    o->pins = c->blks[0].ref;
    o->clock = (int64_t)c->clock;
    return RC_OK;
}

}  // extern "C"
