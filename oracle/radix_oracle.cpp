// Oracle for the radix-tree KV cache: test infrastructure only.
//
// Only the test suite, the package smoke check and the benchmark's CPU-baseline
// leg may load this code.  It shares nothing with the product library: no
// header, no helper, no table.  It is written to be read against the pages:
//
//  * "RadixAttention, eviction and cache churn" (inference-notes note 49),
//    section 2: each edge of the tree holds a run of tokens and the KV of those
//    tokens; lookup walks down one token at a time until a token differs, and
//    there the edge splits into a shared part and two branches; a finished
//    request's whole path, outputs included, stays in the tree.
//  * same note, section 4: the cache and the running requests share one pool;
//    every running request pins its path with a reference count and only
//    nodes whose count is 0 are candidates; leaves go first, least recently
//    used first; a node whose children are all gone becomes a leaf and can be
//    evicted later, so the shared trunk lives longest.
//  * same note, section 5: requests can be served longest-cached-prefix-first
//    (arrival order otherwise).
//  * the unite.ai article on SGLang, RadixAttention paragraph and the
//    nine-step walkthrough: an LRU cache of KV kept in a radix tree used for
//    match, insert and evict; each new chat turn becomes a new node.
//
// Readings where the pages leave a step open (each one is also listed in the
// design notes):
//  - an insert adds at most one new node (the unmatched tail); nodes are split
//    at divergence and never merged;
//  - a match that ends inside a run splits the run, so a pinned prefix ends on
//    a node boundary; an insert splits likewise where it diverges or ends; the
//    new upper node takes the lower node's reference count and is stamped now;
//  - the LRU clock is a counter that each match and each insert advance by
//    one; every node on the touched path (root included) takes the new value;
//    the scheduler's look-ahead touches nothing;
//  - eviction removes whole leaves with count 0, never the root, in order of
//    (last access, node id); it stops as soon as the freed count reaches the
//    request, or when no candidate is left; a parent that becomes a childless
//    count-0 node is a candidate within the same call;
//  - the allocator hands out the n smallest free slot ids in ascending order;
//  - node ids count node creations from 0 (the root); a split gives the new
//    upper node the next id, the lower node keeps its id;
//  - the longest-prefix-first order sorts by the current look-ahead match
//    length, longest first, ties by arrival.
//
// Everything here is deliberately naive: std::map children, a std::set free
// list, and a full scan of all nodes to find each eviction victim.

#include <cstdint>
#include <cstdio>
#include <cstring>
#include <map>
#include <set>
#include <string>
#include <vector>
#include <algorithm>

namespace {

enum : int { O_OK = 0, O_ARG = -1, O_NOMEM = -2, O_STATE = -3 };
enum : uint8_t { SLOT_FREE = 0, SLOT_CALLER = 1, SLOT_TREE = 2 };

struct Node {
    int64_t id = 0;
    Node* parent = nullptr;
    std::vector<int32_t> tokens;
    std::vector<int32_t> slots;
    std::map<int32_t, Node*> children;  // keyed by the first token of the child's run
    int64_t ref = 0;
    uint64_t last_access = 0;
};

struct Tree {
    int64_t pool = 0;
    std::vector<uint8_t> state;          // per slot: free / held by a caller / in the tree
    std::set<int32_t> free_slots;
    Node* root = nullptr;
    std::map<int64_t, Node*> by_id;
    uint64_t clock = 0;
    int64_t next_id = 0;
    // statistics
    int64_t match_calls = 0, match_tokens = 0, match_hits = 0, match_hit_tokens = 0;
    int64_t insert_calls = 0, insert_new_tokens = 0, insert_dup_freed = 0;
    int64_t evicted_nodes = 0, evicted_tokens = 0;
};

Node* make_node(Tree& t, Node* parent) {
    Node* n = new Node();
    n->id = t.next_id++;
    n->parent = parent;
    t.by_id[n->id] = n;
    return n;
}

// Split node x after its first k tokens; the new node above x holds those k.
Node* split(Tree& t, Node* x, size_t k) {
    Node* up = make_node(t, x->parent);
    up->tokens.assign(x->tokens.begin(), x->tokens.begin() + k);
    up->slots.assign(x->slots.begin(), x->slots.begin() + k);
    x->tokens.erase(x->tokens.begin(), x->tokens.begin() + k);
    x->slots.erase(x->slots.begin(), x->slots.begin() + k);
    x->parent->children[up->tokens[0]] = up;
    up->children[x->tokens[0]] = x;
    x->parent = up;
    up->ref = x->ref;
    up->last_access = t.clock;
    return up;
}

// Walk down from the root along tok[0..n).  Returns the number of matched
// tokens.  With do_split, a walk that stops inside a run splits it so that
// the matched part ends on a node; `path` then lists root..end.  Without it,
// nothing changes and `slots_out` (if given) receives the matched slots.
int64_t walk(Tree& t, const int32_t* tok, int64_t n, bool do_split,
             std::vector<Node*>* path, std::vector<int32_t>* slots_out) {
    Node* cur = t.root;
    if (path) path->push_back(cur);
    int64_t i = 0;
    while (i < n) {
        auto it = cur->children.find(tok[i]);
        if (it == cur->children.end()) break;
        Node* c = it->second;
        size_t k = 0;
        while (k < c->tokens.size() && i + (int64_t)k < n && c->tokens[k] == tok[i + k]) ++k;
        if (slots_out) slots_out->insert(slots_out->end(), c->slots.begin(), c->slots.begin() + k);
        i += (int64_t)k;
        if (k < c->tokens.size()) {
            if (do_split) {
                c = split(t, c, k);
                if (path) path->push_back(c);
            }
            break;
        }
        cur = c;
        if (path) path->push_back(cur);
    }
    return i;
}

void stamp(Tree& t, const std::vector<Node*>& path) {
    for (Node* p : path) p->last_access = t.clock;
}

std::vector<int32_t> path_slots(const std::vector<Node*>& path) {
    std::vector<int32_t> s;
    for (Node* p : path) s.insert(s.end(), p->slots.begin(), p->slots.end());
    return s;
}

bool is_leaf_candidate(const Tree& t, const Node* n) {
    return n != t.root && n->children.empty() && n->ref == 0;
}

void dump_node(const Node* n, std::string& out) {
    char buf[96];
    std::snprintf(buf, sizeof buf, "%lld %lld %lld %llu %zu:", (long long)n->id,
                  (long long)(n->parent ? n->parent->id : -1), (long long)n->ref,
                  (unsigned long long)n->last_access, n->tokens.size());
    out += buf;
    for (int32_t v : n->tokens) { out += ' '; out += std::to_string(v); }
    out += " |";
    for (int32_t v : n->slots) { out += ' '; out += std::to_string(v); }
    out += '\n';
    for (auto& kv : n->children) dump_node(kv.second, out);
}

void delete_all(Node* n) {
    for (auto& kv : n->children) delete_all(kv.second);
    delete n;
}

}  // namespace

extern "C" {

void* oracle_tree_new(int64_t pool_slots) {
    if (pool_slots < 0 || pool_slots > INT32_MAX) return nullptr;
    Tree* t = new Tree();
    t->pool = pool_slots;
    t->state.assign((size_t)pool_slots, SLOT_FREE);
    for (int64_t s = 0; s < pool_slots; ++s) t->free_slots.insert((int32_t)s);
    t->root = make_node(*t, nullptr);
    return t;
}

void oracle_tree_free(void* h) {
    Tree* t = (Tree*)h;
    if (!t) return;
    delete_all(t->root);
    delete t;
}

// Longest cached prefix of tok[0..n); optionally pins root..end.
int oracle_match(void* h, const int32_t* tok, int64_t n, int pin,
                 int64_t* matched, int32_t* out_slots, int64_t* node) {
    Tree& t = *(Tree*)h;
    if (n < 0 || (n > 0 && !tok)) return O_ARG;
    t.clock += 1;
    std::vector<Node*> path;
    int64_t m = walk(t, tok, n, true, &path, nullptr);
    stamp(t, path);
    if (pin) for (Node* p : path) p->ref += 1;
    if (out_slots) {
        std::vector<int32_t> s = path_slots(path);
        std::copy(s.begin(), s.end(), out_slots);
    }
    if (matched) *matched = m;
    if (node) *node = path.back()->id;
    t.match_calls += 1;
    t.match_tokens += n;
    t.match_hit_tokens += m;
    if (m > 0) t.match_hits += 1;
    return O_OK;
}

// Insert tok[0..n) with the caller's slots.  Slots of the part already in the
// tree that differ from the tree's own go back to the free pool.
int oracle_insert(void* h, const int32_t* tok, const int32_t* slots, int64_t n, int pin,
                  int64_t* present, int64_t* node, int32_t* out_slots) {
    Tree& t = *(Tree*)h;
    if (n < 0 || (n > 0 && (!tok || !slots))) return O_ARG;
    for (int64_t i = 0; i < n; ++i)
        if (slots[i] < 0 || slots[i] >= t.pool) return O_ARG;
    // look first, change nothing until the caller's slots are known to be valid
    std::vector<int32_t> tree_slots;
    int64_t m = walk(t, tok, n, false, nullptr, &tree_slots);
    std::set<int32_t> seen;
    for (int64_t i = 0; i < n; ++i) {
        bool same_as_tree = i < m && slots[i] == tree_slots[(size_t)i];
        if (same_as_tree) continue;
        if (t.state[(size_t)slots[i]] != SLOT_CALLER) return O_STATE;
        if (!seen.insert(slots[i]).second) return O_STATE;
    }
    t.clock += 1;
    std::vector<Node*> path;
    int64_t m2 = walk(t, tok, n, true, &path, nullptr);
    (void)m2;
    if (m < n) {
        Node* leaf = make_node(t, path.back());
        leaf->tokens.assign(tok + m, tok + n);
        leaf->slots.assign(slots + m, slots + n);
        path.back()->children[leaf->tokens[0]] = leaf;
        for (int32_t s : leaf->slots) t.state[(size_t)s] = SLOT_TREE;
        path.push_back(leaf);
    }
    int64_t dup = 0;
    for (int64_t i = 0; i < m; ++i) {
        if (slots[i] != tree_slots[(size_t)i]) {
            t.state[(size_t)slots[i]] = SLOT_FREE;
            t.free_slots.insert(slots[i]);
            dup += 1;
        }
    }
    stamp(t, path);
    if (pin) for (Node* p : path) p->ref += 1;
    if (out_slots) {
        for (int64_t i = 0; i < n; ++i) out_slots[i] = i < m ? tree_slots[(size_t)i] : slots[i];
    }
    if (present) *present = m;
    if (node) *node = path.back()->id;
    t.insert_calls += 1;
    t.insert_new_tokens += n - m;
    t.insert_dup_freed += dup;
    return O_OK;
}

// Drop one pin of the path root..node.
int oracle_release(void* h, int64_t node_id) {
    Tree& t = *(Tree*)h;
    auto it = t.by_id.find(node_id);
    if (it == t.by_id.end()) return O_STATE;
    Node* n = it->second;
    if (n->ref <= 0) return O_STATE;
    for (Node* p = n; p; p = p->parent) p->ref -= 1;
    return O_OK;
}

// Evict unpinned leaves, least recently used first, until >= n_tokens freed.
int oracle_evict(void* h, int64_t n_tokens, int64_t* freed, int64_t* log, int64_t log_cap,
                 int64_t* n_evicted) {
    Tree& t = *(Tree*)h;
    if (n_tokens < 0) return O_ARG;
    int64_t got = 0, count = 0;
    while (got < n_tokens) {
        Node* victim = nullptr;
        for (auto& kv : t.by_id) {
            Node* c = kv.second;
            if (!is_leaf_candidate(t, c)) continue;
            if (!victim || c->last_access < victim->last_access ||
                (c->last_access == victim->last_access && c->id < victim->id))
                victim = c;
        }
        if (!victim) break;
        for (int32_t s : victim->slots) {
            t.state[(size_t)s] = SLOT_FREE;
            t.free_slots.insert(s);
        }
        got += (int64_t)victim->slots.size();
        victim->parent->children.erase(victim->tokens[0]);
        t.by_id.erase(victim->id);
        if (log && count < log_cap) log[count] = victim->id;
        count += 1;
        t.evicted_nodes += 1;
        t.evicted_tokens += (int64_t)victim->slots.size();
        delete victim;
    }
    if (freed) *freed = got;
    if (n_evicted) *n_evicted = count;
    return O_OK;
}

int oracle_alloc(void* h, int64_t n, int32_t* out) {
    Tree& t = *(Tree*)h;
    if (n < 0 || (n > 0 && !out)) return O_ARG;
    if ((int64_t)t.free_slots.size() < n) return O_NOMEM;
    for (int64_t i = 0; i < n; ++i) {
        int32_t s = *t.free_slots.begin();
        t.free_slots.erase(t.free_slots.begin());
        t.state[(size_t)s] = SLOT_CALLER;
        out[i] = s;
    }
    return O_OK;
}

int oracle_free(void* h, const int32_t* slots, int64_t n) {
    Tree& t = *(Tree*)h;
    if (n < 0 || (n > 0 && !slots)) return O_ARG;
    std::set<int32_t> seen;
    for (int64_t i = 0; i < n; ++i) {
        if (slots[i] < 0 || slots[i] >= t.pool) return O_ARG;
        if (t.state[(size_t)slots[i]] != SLOT_CALLER || !seen.insert(slots[i]).second) return O_STATE;
    }
    for (int64_t i = 0; i < n; ++i) {
        t.state[(size_t)slots[i]] = SLOT_FREE;
        t.free_slots.insert(slots[i]);
    }
    return O_OK;
}

// policy 0 = arrival order, 1 = longest cached prefix first (ties by arrival).
int oracle_sched_order(void* h, int policy, const int32_t* flat_tokens, const int64_t* lens,
                       int32_t n, int32_t* out) {
    Tree& t = *(Tree*)h;
    if (n < 0 || (n > 0 && (!lens || !out)) || (policy != 0 && policy != 1)) return O_ARG;
    std::vector<int64_t> peek((size_t)n, 0);
    int64_t off = 0;
    for (int32_t i = 0; i < n; ++i) {
        if (lens[i] < 0) return O_ARG;
        peek[(size_t)i] = walk(t, flat_tokens + off, lens[i], false, nullptr, nullptr);
        off += lens[i];
    }
    std::vector<int32_t> order((size_t)n);
    for (int32_t i = 0; i < n; ++i) order[(size_t)i] = i;
    if (policy == 1)
        std::stable_sort(order.begin(), order.end(),
                         [&](int32_t a, int32_t b) { return peek[(size_t)a] > peek[(size_t)b]; });
    std::copy(order.begin(), order.end(), out);
    return O_OK;
}

// One scheduling round, in the order the pages give its steps:
//  1. the pending prompts are ordered, longest cached prefix first or by
//     arrival (note 49, section 5);
//  2. in that order each request looks up its prompt and pins the matched
//     path, since a running request holds its path (section 4);
//  3. a request that will decode recomputes at least its last prompt token,
//     so that one new token carries the query: its first computed position is
//     min(matched, prompt_len - 1) (prefill-only requests start at matched);
//  4. it needs slots for every position it will compute: the uncached prompt
//     tail plus max_new decode tokens;
//  5. when fewer slots are free, least-recently-used unpinned leaves are
//     evicted for the shortfall (section 4: cache and running requests share
//     one pool, eviction makes room);
//  6. if the slots still cannot be had, the request drops its pin and the
//     round ends there: no later request overtakes it; the round also ends
//     when max_batch requests (> 0) are in.
// Token rows: row i of the flat arrays starts at the sum over j < i of
// prompt_len[j] + max_new[j] and holds the prompt (only the prompt is read
// here).  slots row i receives the matched slots for positions [0, first)
// and the new ones for [first, prompt_len + max_new).  out_order lists the
// admitted requests in admission order.
int oracle_admit(void* h, int policy, const int32_t* flat_tokens, const int64_t* prompt_len,
                 const int64_t* max_new, int32_t n, int32_t max_batch, int32_t* out_order,
                 int32_t* n_admitted, int64_t* matched, int64_t* first_pos, int64_t* node,
                 int32_t* slots) {
    Tree& t = *(Tree*)h;
    if (n < 0 || !n_admitted || (n > 0 && (!prompt_len || !max_new || !out_order || !matched ||
                                           !first_pos || !node || !slots)))
        return O_ARG;
    *n_admitted = 0;
    std::vector<int64_t> row_off((size_t)n + 1, 0);
    for (int32_t i = 0; i < n; ++i) {
        if (prompt_len[i] < 0 || max_new[i] < 0 || (max_new[i] > 0 && prompt_len[i] == 0)) return O_ARG;
        row_off[(size_t)i + 1] = row_off[(size_t)i] + prompt_len[i] + max_new[i];
        node[i] = -1;
        matched[i] = 0;
        first_pos[i] = 0;
    }
    // step 1 (the ordering reads prompts only: gather them)
    std::vector<int32_t> prompts;
    for (int32_t i = 0; i < n; ++i)
        prompts.insert(prompts.end(), flat_tokens + row_off[(size_t)i], flat_tokens + row_off[(size_t)i] + prompt_len[i]);
    std::vector<int32_t> order((size_t)n);
    int st = oracle_sched_order(h, policy, prompts.data(), prompt_len, n, order.data());
    if (st != O_OK) return st;
    int32_t count = 0;
    for (int32_t k = 0; k < n; ++k) {
        if (max_batch > 0 && count >= max_batch) break;
        const int32_t i = order[(size_t)k];
        const int32_t* tok = flat_tokens + row_off[(size_t)i];
        const int64_t len = prompt_len[i];
        // step 2
        std::vector<int32_t> mslots((size_t)std::max<int64_t>(len, 1));
        int64_t m = 0, nd = -1;
        st = oracle_match(h, tok, len, 1, &m, mslots.data(), &nd);
        if (st != O_OK) return st;
        // steps 3 and 4
        const int64_t first = max_new[i] > 0 ? std::min<int64_t>(m, len - 1) : m;
        const int64_t need = len - first + max_new[i];
        // step 5
        const int64_t free_now = (int64_t)t.free_slots.size();
        if (free_now < need) {
            int64_t freed = 0, cnt = 0;
            st = oracle_evict(h, need - free_now, &freed, nullptr, 0, &cnt);
            if (st != O_OK) return st;
        }
        // step 6
        std::vector<int32_t> fresh((size_t)std::max<int64_t>(need, 1));
        st = oracle_alloc(h, need, fresh.data());
        if (st == O_NOMEM) {
            st = oracle_release(h, nd);
            if (st != O_OK) return st;
            break;
        }
        if (st != O_OK) return st;
        int32_t* row = slots + row_off[(size_t)i];
        for (int64_t j = 0; j < first; ++j) row[j] = mslots[(size_t)j];
        for (int64_t j = 0; j < need; ++j) row[first + j] = fresh[(size_t)j];
        matched[i] = m;
        first_pos[i] = first;
        node[i] = nd;
        out_order[count++] = i;
    }
    *n_admitted = count;
    return O_OK;
}

// The inserts around a batch's run (note 49, section 2: a prompt, once
// computed, is in the tree so concurrent requests can share it; a finished
// request's whole path, outputs included, stays cached).  Rows as in
// oracle_admit, for the n requests of this call; node[i] is the pin the
// request holds and is updated.
//  mode 0, after prefill: insert the prompt with the row's slots (pinned if
//    the request will decode), drop the admission pin, and take the tree's
//    slots for the prompt (the caller's duplicates went back to the pool);
//  mode 1, at finish (requests that decoded): insert prompt + generated
//    tokens unpinned, drop the request's pin.
int oracle_commit(void* h, int mode, const int32_t* flat_tokens, const int64_t* prompt_len,
                  const int64_t* max_new, int32_t n, int32_t* slots, int64_t* node) {
    if (n < 0 || (mode != 0 && mode != 1) || (n > 0 && (!flat_tokens || !prompt_len || !max_new || !slots || !node)))
        return O_ARG;
    int64_t off = 0;
    for (int32_t i = 0; i < n; ++i) {
        const int64_t row_len = prompt_len[i] + max_new[i];
        const int32_t* tok = flat_tokens + off;
        int32_t* row = slots + off;
        off += row_len;
        if (mode == 1 && max_new[i] == 0) continue;
        const int64_t len = mode == 0 ? prompt_len[i] : row_len;
        const int pin = mode == 0 && max_new[i] > 0;
        int64_t present = 0, nd = -1;
        int st = oracle_insert(h, tok, row, len, pin, &present, &nd, row);
        if (st != O_OK) return st;
        st = oracle_release(h, node[i]);
        if (st != O_OK) return st;
        node[i] = pin ? nd : -1;
    }
    return O_OK;
}

// Text dump: one line per node in depth-first order, children by first token:
// "id parent ref last_access ntok: tokens... | slots...".  Returns the length.
int64_t oracle_dump(void* h, char* buf, int64_t cap) {
    Tree& t = *(Tree*)h;
    std::string s;
    dump_node(t.root, s);
    if (buf && cap > 0) {
        int64_t k = std::min<int64_t>(cap - 1, (int64_t)s.size());
        std::memcpy(buf, s.data(), (size_t)k);
        buf[k] = 0;
    }
    return (int64_t)s.size();
}

// Statistics in a fixed order; see the binding for the field names.
int oracle_stats(void* h, int64_t* out) {
    Tree& t = *(Tree*)h;
    int64_t tree_tokens = 0, caller = 0;
    for (auto& kv : t.by_id) tree_tokens += (int64_t)kv.second->slots.size();
    for (uint8_t s : t.state) caller += (s == SLOT_CALLER);
    int64_t v[16] = {
        t.pool, (int64_t)t.free_slots.size(), caller, tree_tokens, (int64_t)t.by_id.size(),
        t.match_calls, t.match_tokens, t.match_hits, t.match_hit_tokens,
        t.insert_calls, t.insert_new_tokens, t.insert_dup_freed,
        t.evicted_nodes, t.evicted_tokens, t.root->ref, (int64_t)t.clock,
    };
    std::memcpy(out, v, sizeof v);
    return O_OK;
}

}  // extern "C"
