// The shared KV pool's slot allocator, used by both host caches (the radix
// tree and the 16-token block comparator).  "RadixAttention, eviction and
// cache churn" (inference-notes note 49), section 4: the cache and the running
// requests draw on one memory pool.
//
// Every slot is FREE, HELD (by a caller: allocated and not yet handed to a
// cache) or CACHED (owned by a cache).  Free slots are a two-level bitmap, so
// "the n smallest free ids, ascending" is a scan of set bits from the lowest
// non-empty word.  Per-slot epoch marks give O(n) duplicate checks.
#pragma once

#include <algorithm>
#include <cstdint>
#include <vector>

namespace rc_pool {

enum : uint8_t { FREE = 0, HELD = 1, CACHED = 2 };

struct SlotPool {
    int64_t pool = 0;
    std::vector<uint8_t> owner;      // per slot: FREE, HELD, CACHED
    std::vector<uint64_t> bits;      // 1 = free
    std::vector<uint64_t> summary;   // 1 = bits[w] != 0
    int64_t n_free = 0, n_held = 0, n_cached = 0;
    std::vector<uint32_t> mark;      // per slot epoch marks for duplicate checks
    uint32_t epoch = 0;

    // All slots free.  May throw std::bad_alloc.
    void init_slots(int64_t pool_slots) {
        pool = pool_slots;
        owner.assign((size_t)pool_slots, FREE);
        mark.assign((size_t)pool_slots, 0);
        size_t nw = (size_t)((pool_slots + 63) / 64);
        bits.assign(nw, ~0ull);
        if (pool_slots & 63) bits[nw - 1] = (1ull << (pool_slots & 63)) - 1;
        summary.assign((nw + 63) / 64 + 1, 0);
        for (size_t w = 0; w < nw; ++w)
            if (bits[w]) summary[w >> 6] |= 1ull << (w & 63);
        n_free = pool_slots;
    }
    void slot_set_free(int32_t s) {
        size_t w = (size_t)s >> 6;
        bits[w] |= 1ull << (s & 63);
        summary[w >> 6] |= 1ull << (w & 63);
    }
    int64_t next_word(int64_t w) const {  // first word index >= w with free bits, or -1
        int64_t nw = (int64_t)bits.size();
        if (w >= nw) return -1;
        size_t sw = (size_t)w >> 6;
        uint64_t m = summary[sw] & (~0ull << (w & 63));
        while (!m) {
            if (++sw >= summary.size()) return -1;
            m = summary[sw];
        }
        return (int64_t)(sw << 6) + __builtin_ctzll(m);
    }
    // The n smallest free ids, ascending, now HELD.  Requires n <= n_free.
    void take_lowest(int64_t n, int32_t* out) {
        int64_t got = 0, w = next_word(0);
        while (got < n) {
            uint64_t b = bits[(size_t)w];
            while (b && got < n) {
                int t = __builtin_ctzll(b);
                b &= b - 1;
                int32_t s = (int32_t)(w * 64 + t);
                out[got++] = s;
                owner[(size_t)s] = HELD;
            }
            bits[(size_t)w] = b;
            if (!b) summary[(size_t)w >> 6] &= ~(1ull << (w & 63));
            if (got < n) w = next_word(w + 1);
        }
        n_free -= n;
        n_held += n;
    }
    // A fresh mark value: mark[s] == epoch means "seen in this check".
    uint32_t new_epoch() {
        if (++epoch == 0) {
            std::fill(mark.begin(), mark.end(), 0);
            epoch = 1;
        }
        return epoch;
    }
    // A HELD or CACHED slot back to the free set.
    void release_slot(int32_t s) {
        uint8_t& o = owner[(size_t)s];
        if (o == HELD) n_held -= 1;
        else if (o == CACHED) n_cached -= 1;
        else return;
        o = FREE;
        slot_set_free(s);
        n_free += 1;
    }
    // A HELD slot handed to a cache.
    void cache_slot(int32_t s) {
        owner[(size_t)s] = CACHED;
        n_held -= 1;
        n_cached += 1;
    }
    // The caller's free of HELD slots: -1 if an id is out of range, -2 if one
    // is not HELD or repeats (nothing changes then), 0 after freeing them all.
    int free_held(const int32_t* slots, int64_t n) {
        for (int64_t i = 0; i < n; ++i)
            if (slots[i] < 0 || slots[i] >= pool) return -1;
        const uint32_t e = new_epoch();
        for (int64_t i = 0; i < n; ++i) {
            int32_t s = slots[i];
            if (owner[(size_t)s] != HELD || mark[(size_t)s] == e) return -2;
            mark[(size_t)s] = e;
        }
        for (int64_t i = 0; i < n; ++i) release_slot(slots[i]);
        return 0;
    }
};

}  // namespace rc_pool
