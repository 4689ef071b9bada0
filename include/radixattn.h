/* radixattn.h: C ABI of the prefix-shared radix-tree KV cache and its kernels.
 *
 * Two halves.
 *
 *  Host (radix tree, reference counts, LRU, slot allocator, scheduling order):
 *  rc_create, rc_destroy, rc_match_prefix, rc_insert, rc_release, rc_evict,
 *  rc_alloc, rc_free, sched_order, rc_stats, rc_dump.  Plain C++ on the
 *  caller's thread; not thread-safe per cache object.
 *
 *  Device (hand-written CUDA for sm_103a): kv_store, attn_decode, attn_extend,
 *  their workspace queries, and rc_sync.  All device memory is the caller's:
 *  the library never allocates it (its one device array is the fixed scratch
 *  of attn_decode_static).  Device calls enqueue work on `stream` and
 *  return; an error detected inside a kernel (a slot index outside the pool)
 *  is OR-ed into the caller's device error word and read back by rc_sync.
 *
 * The pages this follows:
 *  [N49] "RadixAttention, eviction and cache churn" (inference-notes note 49):
 *        section 2 (edges hold token runs and their KV; lookup walks one token
 *        at a time; the edge splits at the first differing token; finished
 *        requests, outputs included, stay cached), section 4 (shared pool;
 *        reference-count pinning; unpinned least-recently-used leaves evicted
 *        first; a parent whose children are gone becomes a leaf), section 5
 *        (longest cached prefix first vs arrival order).
 *  [SG]  unite.ai article on SGLang: the RadixAttention paragraph (an LRU
 *        cache of KV in a radix tree for match, insert and evict) and the
 *        nine-step walkthrough of the tree.
 *  [LMI] SageMaker LMI / Falcon article, "prefill and decode phases": prefill
 *        runs the whole prompt at once; decode produces one token per step
 *        from the cached K/V.
 *  [DS]  SGLang engineering article, section 1 (MLA): a single KV head whose
 *        decode kernel serves several query heads per block to cut KV traffic.
 *
 * Conventions.  Token ids and slot ids are int32.  A slot is one row of the
 * KV pool: for grouped-query attention the pool holds K and V as
 * [n_slots][kv_heads][head_dim] bf16 each; for the latent (MLA) layout one
 * array [n_slots][head_dim_k] bf16 whose first head_dim_v columns are V.
 * Every status is an rc_status; nothing aborts and no C++ exception crosses
 * this boundary.
 */
#ifndef RADIXATTN_H
#define RADIXATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t rc_status;
#define RC_OK               0
#define RC_ERR_ARG         -1  /* bad argument: null pointer, negative size, id out of range */
#define RC_ERR_NOMEM       -2  /* not enough free slots (rc_alloc never evicts by itself) */
#define RC_ERR_STATE       -3  /* unknown or unpinned node, slot not owned by the caller */
#define RC_ERR_CUDA        -4  /* a CUDA runtime call failed */
#define RC_ERR_TIMEOUT     -5  /* a bounded device wait gave up */
#define RC_ERR_DEVICE      -6  /* a kernel found a slot index outside the pool */
#define RC_ERR_UNSUPPORTED -7  /* head layout this build has no kernel for */
#define RC_ERR_SCRATCH     -8  /* needs more than the library's fixed scratch area */

/* Scheduling policies of sched_order. */
#define RC_FCFS 0  /* arrival order */
#define RC_LPM  1  /* longest cached prefix first, ties by arrival [N49 s.5] */

typedef struct rc_cache rc_cache;   /* opaque host object */
typedef int64_t rc_node;            /* node id: 0 is the root; ids count node creations */
typedef struct CUstream_st* rc_stream_t;  /* a cudaStream_t; NULL = legacy default stream */

/* ------------------------------------------------------------------ host */

/* Create a cache over a pool of `pool_slots` slots (ids 0..pool_slots-1), all
 * free [N49 s.4: the cache and the running requests share one pool of KV
 * slots].  `pool_slots` in [0, 2^31-1].  *out receives the handle.
 * Errors: RC_ERR_ARG (bad size or null out), RC_ERR_NOMEM (host allocation). */
rc_status rc_create(int64_t pool_slots, rc_cache** out);
void rc_destroy(rc_cache* cache);

/* Longest cached prefix of tok[0..n) [N49 s.2: lookup walks down one token at a
 * time until a token differs].  A match that ends inside an edge splits that
 * edge so the prefix ends on a node; the new upper node takes the lower node's
 * reference count.  Advances the LRU clock by one and stamps every node on the
 * path root..end.  With pin != 0 every node on that path gets one more
 * reference [N49 s.4]; undo with rc_release(*out_node).
 * out_slots: NULL or room for n slot ids; receives the matched prefix's slots.
 * *matched: matched length.  *out_node: end node (root when nothing matched).
 * Errors: RC_ERR_ARG (n < 0, null tok with n > 0, null matched/out_node). */
rc_status rc_match_prefix(rc_cache* cache, const int32_t* tok, int64_t n, int pin,
                          int64_t* matched, int32_t* out_slots, rc_node* out_node);

/* Insert tok[0..n) whose K/V sit in slots[0..n) [N49 s.2: a finished request's
 * path stays cached; SG walkthrough: a new turn becomes a new node].  At most
 * one node is added (the unmatched tail); an edge is split where the new
 * sequence leaves it or ends inside it.  Ownership: the slots of the new tail
 * must be held by the caller (from rc_alloc) and pass to the tree; for the
 * already-present part, a caller slot equal to the tree's slot at that
 * position is left alone and any other caller slot goes back to the free
 * pool (a duplicate).  Validation happens before any change: on error nothing
 * changed.  Advances the LRU clock by one and stamps the path; pins the path
 * root..end when pin != 0.
 * *already_present: length of the part that was already cached.
 * out_slots: NULL or room for n; receives the tree's slots for every position
 * (what the caller's slot table should hold from now on).
 * Errors: RC_ERR_ARG (bad sizes/pointers, slot id out of range), RC_ERR_STATE
 * (a slot that should be the caller's is free or in the tree, or repeats). */
rc_status rc_insert(rc_cache* cache, const int32_t* tok, const int32_t* slots, int64_t n,
                    int pin, int64_t* already_present, rc_node* out_node, int32_t* out_slots);

/* Drop one reference from every node on the path root..node [N49 s.4].
 * Errors: RC_ERR_STATE (unknown or evicted node, or node not pinned). */
rc_status rc_release(rc_cache* cache, rc_node node);

/* Evict unpinned leaves, least recently used first (ties: lower node id),
 * until at least n_tokens slots are freed or no candidate is left [N49 s.4;
 * SG walkthrough steps 5, 8, 9].  Whole leaves only, never the root; a parent
 * left without children and without pins becomes a candidate in the same call.
 * *freed: slots freed (may be < n_tokens).  log: NULL or room for log_cap node
 * ids, in eviction order; *n_evicted: nodes evicted (even beyond log_cap).
 * Errors: RC_ERR_ARG (n_tokens < 0, null freed or n_evicted). */
rc_status rc_evict(rc_cache* cache, int64_t n_tokens, int64_t* freed,
                   int64_t* log, int64_t log_cap, int64_t* n_evicted);

/* Take the n smallest free slot ids, ascending, into out[0..n) [N49 s.4: the
 * cache and the running requests share one pool].  Never evicts.
 * Errors: RC_ERR_ARG, RC_ERR_NOMEM (fewer than n free; nothing taken). */
rc_status rc_alloc(rc_cache* cache, int64_t n, int32_t* out);

/* Give caller-held slots back to the pool [N49 s.4: one shared pool; slots a
 * request took and will not insert return to it].  Errors: RC_ERR_ARG (id out
 * of range), RC_ERR_STATE (slot not held by the caller, or repeated). */
rc_status rc_free(rc_cache* cache, const int32_t* slots, int64_t n);

/* Serving order of n pending prompts [N49 s.5].  RC_FCFS: 0..n-1.
 * RC_LPM: by the length each prompt would match now, longest first, ties by
 * index; the look-ahead changes nothing (no split, stamp or pin).
 * prompts: n host pointers; lens: n lengths.  out_order: room for n.
 * Errors: RC_ERR_ARG. */
rc_status sched_order(rc_cache* cache, int policy, const int32_t* const* prompts,
                      const int64_t* lens, int32_t n, int32_t* out_order);

/* One request for the batched calls below.  tokens: host buffer holding the
 * prompt (prompt_len tokens) followed, by the time rc_commit(RC_COMMIT_FINISH)
 * runs, by the max_new generated tokens.  slots: caller buffer of
 * prompt_len + max_new entries that rc_admit fills and rc_commit updates.
 * The remaining fields are outputs. */
typedef struct rc_request {
    const int32_t* tokens;
    int64_t prompt_len;
    int64_t max_new;
    int32_t* slots;
    int64_t matched;   /* cached prefix found at admission */
    int64_t first;     /* first position the prefill computes */
    rc_node node;      /* node the request holds a pin on (-1: none) */
    int32_t admitted;
} rc_request;

/* Admission of one scheduling round, natively: sched_order(policy), then in
 * that order rc_match_prefix(pin), first = min(matched, prompt_len - 1) for a
 * request that will decode (one new token carries the query) else matched,
 * rc_alloc(prompt_len - first + max_new) with rc_evict of the shortfall on
 * RC_ERR_NOMEM; a request that still does not fit is unpinned and stops
 * admission for the round (no overtaking), as does reaching max_batch
 * (<= 0: no limit) [N49 s.4, s.5].  slots[0..first) = the matched slots,
 * slots[first..) = the new ones, in allocation order.  out_order receives the
 * indices of the admitted requests in admission order; *n_admitted their count.
 * Errors: RC_ERR_ARG. */
rc_status rc_admit(rc_cache* cache, int policy, rc_request* reqs, int32_t n, int32_t max_batch,
                   int32_t* out_order, int32_t* n_admitted);

/* Inserts for a batch of admitted requests (indices idx[0..n)).
 * RC_COMMIT_PREFILL: rc_insert(prompt, slots[0..prompt_len)) pinned if the
 *   request will decode, drop the admission pin, slots[0..prompt_len) = the
 *   tree's slots (duplicates were freed) [N49 s.2: only the new part computed].
 * RC_COMMIT_FINISH: rc_insert(prompt + generated, slots) unpinned and drop the
 *   request's pin [N49 s.2: a finished request's path, outputs included,
 *   stays] (requests with max_new == 0 are skipped).
 * The records must be as rc_admit (and, for FINISH, the PREFILL commit) left
 * them: each insert starts at the request's pinned node, so slots[0..first)
 * (PREFILL) and slots[0..prompt_len) (FINISH), which hold the tree's own
 * slots there, are not read again.
 * Errors: RC_ERR_ARG, or the first failing rc_insert / rc_release status
 * (requests before it are committed). */
#define RC_COMMIT_PREFILL 0
#define RC_COMMIT_FINISH  1
rc_status rc_commit(rc_cache* cache, rc_request* reqs, const int32_t* idx, int32_t n, int mode);

/* Cascade segments of a running batch, read off the tree [N49 s.1: the
 * shared parts of layered prompts form a tree]: every node on the pinned path
 * of at least two of the n requests (nodes[i] = request i's pinned node) is a
 * segment, read once for all of them.  Request i's own keys start after the
 * last shared node on its path (a node shared by several requests is shared
 * in full: their matches split edges at every divergence).
 * Outputs (caller buffers): seg_slots (cap seg_slots_cap), seg_indptr (n_seg+1),
 * seg_row_indptr (n_seg+1), seg_rows and req_seg_pos (cap rows_cap),
 * req_seg_indptr (n+1), private_start (n); *n_seg, *n_seg_slots, *total_rows,
 * *max_seg_len, *max_seg_rows.  Segments come in depth-first order of first
 * appearance; rows within a segment ascend.  seg_cap bounds n_seg.
 * Errors: RC_ERR_ARG (bad pointers), RC_ERR_STATE (unknown node),
 * RC_ERR_NOMEM (a buffer is too small). */
rc_status rc_cascade_plan(rc_cache* cache, const rc_node* nodes, int32_t n, int32_t* seg_slots,
                          int64_t seg_slots_cap, int32_t* seg_indptr, int32_t* seg_row_indptr,
                          int32_t* seg_rows, int32_t* req_seg_indptr, int32_t* req_seg_pos,
                          int64_t rows_cap, int64_t* private_start, int32_t seg_cap, int32_t* n_seg,
                          int64_t* n_seg_slots, int32_t* total_rows, int32_t* max_seg_len,
                          int32_t* max_seg_rows);

/* Counters of the cache (a library extra: the pages define the hit rates
 * these counts give [N49 s.6, SG evaluation], not an interface for them).
 * Errors: RC_ERR_ARG (null cache or out). */
typedef struct rc_stats_t {
    int64_t pool_slots, free_slots, caller_slots, tree_tokens, nodes;
    int64_t match_calls, match_tokens, match_hits, match_hit_tokens;
    int64_t insert_calls, insert_new_tokens, insert_dup_freed;
    int64_t evicted_nodes, evicted_tokens;
    int64_t pins;    /* references held on the root = pinned paths */
    int64_t clock;   /* LRU clock */
} rc_stats_t;
rc_status rc_stats(rc_cache* cache, rc_stats_t* out);

/* Text dump of the tree for tests: one line per node, depth first, children
 * in ascending first-token order:
 *   "<id> <parent id or -1> <ref> <last access> <ntok>: <tokens> | <slots>\n"
 * Writes at most cap-1 bytes plus a NUL; *needed = full length (no NUL). */
rc_status rc_dump(rc_cache* cache, char* buf, int64_t cap, int64_t* needed);

/* Keys of an image for the tree [SG, multimodal results: the input image's
 * hash is the key in the radix tree, so its tokens' KV is reused]: a run of
 * n_tokens keys, all in [-2^30, -1] (never a text token id, which is >= 0),
 * a function of the image's bytes alone.  Definition: h = FNV-1a 64 of
 * data[0..bytes); out[i] = -1 - (splitmix64 finaliser of
 * h + (i+1)*0x9E3779B97F4A7C15) >> 34.  Put the run where the image sits in the
 * prompt; equal images give equal runs, so a later prompt with the same image
 * matches through it.  data may be NULL when bytes == 0.
 * Errors: RC_ERR_ARG (negative sizes, null pointers with non-zero sizes). */
rc_status rc_image_key(const void* data, int64_t bytes, int32_t n_tokens, int32_t* out);

/* ---------------------------------------------------------- block comparator
 * A prefix cache over fixed-size token blocks, the scheme [N49 s.3] sets
 * against the radix tree (vLLM: a hash chain of 16-token blocks, whole-block
 * matches, reference counts, least recently used first).  Same pool rules,
 * call shapes, clock and pins as the rc_* calls, so both run one trace and
 * differ only in match granularity.  Readings: only a full block is cached,
 * keyed exactly by (the block before it, its tokens); a lookup walks whole
 * blocks from the start; insert caches the full blocks not cached yet and
 * leaves the partial last block with the caller, who frees it (bc_free) when
 * the request is done; every match and insert advance the clock by one and
 * stamp the touched chain (root included); a pin counts on every block of
 * the chain; eviction takes unpinned blocks (never the root) by last access,
 * ties to the block farther from the chain's start, whole blocks, until the
 * freed count reaches the request.  Node handles (rc_node) are block ids:
 * 0 is the root (the empty chain), ids count block creations. */
typedef struct bc_cache bc_cache;

/* block_tokens in [1, 4096] (16 for the comparison of [N49 s.3]).
 * Errors: RC_ERR_ARG, RC_ERR_NOMEM. */
rc_status bc_create(int64_t pool_slots, int32_t block_tokens, bc_cache** out);
void bc_destroy(bc_cache* cache);
/* As rc_match_prefix; *matched is a multiple of block_tokens, *out_node the
 * last matched block (0 when none). */
rc_status bc_match_prefix(bc_cache* cache, const int32_t* tok, int64_t n, int pin,
                          int64_t* matched, int32_t* out_slots, rc_node* out_node);
/* As rc_insert for the floor(n / block_tokens) full blocks of tok[0..n); the
 * slots of the partial last block stay held by the caller.  *already_present:
 * tokens in blocks that were cached before the call.  out_slots: room for n
 * (cached slots, then the caller's for new blocks and the partial tail).
 * Errors: RC_ERR_ARG, RC_ERR_STATE (nothing changed), RC_ERR_NOMEM. */
rc_status bc_insert(bc_cache* cache, const int32_t* tok, const int32_t* slots, int64_t n,
                    int pin, int64_t* already_present, rc_node* out_node, int32_t* out_slots);
/* Drop one pin from every block of the chain ending at node.
 * Errors: RC_ERR_STATE (unknown or evicted block, or not pinned). */
rc_status bc_release(bc_cache* cache, rc_node node);
/* Evict unpinned blocks until at least n_tokens slots are freed or none is
 * left; log: NULL or room for log_cap block ids in eviction order;
 * *n_evicted counts blocks (even beyond log_cap).  Errors: RC_ERR_ARG. */
rc_status bc_evict(bc_cache* cache, int64_t n_tokens, int64_t* freed,
                   int64_t* log, int64_t log_cap, int64_t* n_evicted);
/* As rc_alloc / rc_free. */
rc_status bc_alloc(bc_cache* cache, int64_t n, int32_t* out);
rc_status bc_free(bc_cache* cache, const int32_t* slots, int64_t n);
/* As sched_order, with the block-granular look-ahead match. */
rc_status bc_sched_order(bc_cache* cache, int policy, const int32_t* const* prompts,
                         const int64_t* lens, int32_t n, int32_t* out_order);
/* As rc_stats: nodes counts live blocks (root included), evicted_nodes blocks. */
rc_status bc_stats(bc_cache* cache, rc_stats_t* out);

/* ---------------------------------------------------------------- device */

/* KV pool in HBM (caller-owned).  GQA: k and v are [n_slots][kv_heads][head_dim]
 * bf16, row-major, 16-byte aligned.  Latent (mla != 0): kv_heads == 1, k is
 * [n_slots][head_dim_k] and its first head_dim_v columns are V; v is NULL.
 * err: device int32 that kernels OR RC error bits into (may be NULL).
 * FP8 pool (kv_fp8 != 0; GQA, head_dim 128) [DS s.1: KV cache FP8 quantisation;
 * block-wise FP8: E4M3 with one dynamic scale per token per 128-channel
 * group]: k and v hold E4M3 codes, one byte per element in the same
 * [n_slots][kv_heads][head_dim] layout, and k_scale / v_scale are fp32
 * [n_slots][kv_heads]; an element's value is its code times the scale of its
 * (slot, head) row.  kv_store quantises (see there); attn_decode reads it. */
typedef struct rc_pool_desc {
    void* k;
    void* v;
    int64_t n_slots;
    int32_t kv_heads;
    int32_t head_dim_k;
    int32_t head_dim_v;
    int32_t mla;
    int32_t* err;
    int32_t kv_fp8;
    float* k_scale;
    float* v_scale;
} rc_pool_desc;

typedef struct rc_attn_desc {
    rc_pool_desc pool;
    int32_t q_heads;   /* multiple of kv_heads; query head h reads kv head h / (q_heads/kv_heads) */
    float sm_scale;    /* scale of q.k inside the softmax */
} rc_attn_desc;

/* Per-request slot tables on the device (caller-owned).  The keys of request b
 * are, in position order, slots[start[b] .. start[b] + len[b]).  Rows may have
 * room to grow (kv_store appends).  max_len: a host-side bound on every len[b]
 * (sizes the grid; longer rows are an error).  table_len: entries in `slots`;
 * a row outside [0, table_len) is not read and flags RC_ERR_DEVICE. */
typedef struct rc_kv_table {
    const int32_t* slots;
    const int32_t* start;
    const int32_t* len;
    int32_t max_len;
    int64_t table_len;
} rc_kv_table;

/* Scatter n new tokens' K/V rows into the pool [N49 s.2: each edge keeps the
 * KV of its tokens].  k_new: [n][kv_heads][head_dim_k] bf16; v_new:
 * [n][kv_heads][head_dim_v] (NULL for the latent layout).  Row i goes to slot
 * slots[i].  If table and table_pos are both non-NULL, also
 * table[table_pos[i]] = slots[i] (appends to the slot tables).
 * A slot outside [0, n_slots) is skipped and flags RC_ERR_DEVICE in pool->err.
 * FP8 pool: each (token, head) row x of head_dim bf16 values is stored as
 * scale = amax|x| / 448 (fp32, rounded to nearest) and codes
 * e4m3(x_i / scale) (fp32 quotient rounded to nearest, then to the nearest
 * E4M3 value, ties to even, saturating at +-448); an all-zero row stores scale
 * 0 and zero codes.
 * Errors (host): RC_ERR_ARG, RC_ERR_UNSUPPORTED (row bytes not a multiple of 16;
 * an FP8 pool that is latent or whose head_dim is not 128), RC_ERR_CUDA (launch). */
rc_status kv_store(const rc_pool_desc* pool, const int32_t* slots, const void* k_new,
                   const void* v_new, int32_t n, int32_t* table, const int32_t* table_pos,
                   rc_stream_t stream);

/* Shared-prefix segments for cascade decode (all device arrays caller-owned;
 * the tree gives them: a node pinned by several running requests is one
 * segment) [N49 s.1: prompts share in layers, so the shared parts form a tree].
 * Segment s covers keys seg_slots[seg_indptr[s] .. seg_indptr[s+1]) and is
 * read once for every batch row listed in seg_rows[seg_row_indptr[s] ..
 * seg_row_indptr[s+1]).  The inverse map lists, for batch row b, the
 * positions p in seg_rows with seg_rows[p] == b:
 * req_seg_pos[req_seg_indptr[b] .. req_seg_indptr[b+1]).  With a cascade, the
 * kv table of attn_decode holds only each row's remaining (private) keys; the
 * result equals flat decode over segments + private keys.  max_seg_len and
 * max_seg_rows are host bounds on keys and rows per segment (they size the
 * grid); total_seg_rows = seg_row_indptr[n_seg].
 * host_seg_indptr, host_seg_row_indptr: NULL, or HOST copies of seg_indptr
 * and seg_row_indptr (n_seg + 1 entries each, equal to the device arrays,
 * read by the call itself).  With them the cascade grid has one CTA per
 * non-empty (segment, key chunk, row block) only; without them it spans
 * max_seg_rows x max_seg_len for every segment and the CTAs past a short
 * segment's rows or keys leave at once (a library convenience: the pages
 * describe the shared layers, not a launch grid). */
typedef struct rc_cascade {
    int32_t n_seg;
    const int32_t* seg_slots;
    const int32_t* seg_indptr;
    const int32_t* seg_row_indptr;
    const int32_t* seg_rows;
    const int32_t* req_seg_indptr;
    const int32_t* req_seg_pos;
    int32_t max_seg_len;
    int32_t max_seg_rows;
    int32_t total_seg_rows;
    const int32_t* host_seg_indptr;
    const int32_t* host_seg_row_indptr;
} rc_cascade;

/* Workspace bytes attn_decode needs for this batch (split partials). */
rc_status attn_decode_workspace(const rc_attn_desc* desc, int32_t batch, int32_t max_len,
                                const rc_cascade* cascade, size_t* bytes);

/* One decode step for `batch` requests [LMI decode phase; N49 s.2]: row b's
 * single query q[b] ([batch][q_heads][head_dim_k] bf16) sits at the last
 * position of its context and attends to all of it:
 *   out[b][h] = sum_j softmax_j(sm_scale * q[b][h].K[j][g(h)]) V[j][g(h)]
 * over the cascade segments of row b (if any) and then its table row.
 * out: [batch][q_heads][head_dim_v] bf16.  lse: NULL or [batch][q_heads] fp32,
 * natural log of the softmax denominator.  ws: attn_decode_workspace bytes.
 * Errors: RC_ERR_ARG, RC_ERR_UNSUPPORTED (head layout), RC_ERR_CUDA. */
rc_status attn_decode(const rc_attn_desc* desc, const void* q, const rc_kv_table* kv,
                      int32_t batch, const rc_cascade* cascade, void* out, float* lse,
                      void* ws, size_t ws_bytes, rc_stream_t stream);

/* attn_decode for a step whose new token's K/V is not stored yet: kv_store of
 * those rows followed by attn_decode, in one launch less [N49 s.2: the new
 * token's K/V joins its request's edge; LMI decode phase].  k_new, v_new:
 * [batch][kv_heads][head_dim] bf16, 16-byte aligned, the K/V of each row's
 * last key (position len[b]-1, slot slots[start[b]+len[b]-1]).  The kernel
 * that reads row b's last key writes k_new[b]/v_new[b] to that slot of the
 * pool and uses them directly for that key; the result (out, lse) is that of
 * attn_decode on the updated pool, bit for bit.  The last key must be in the
 * row's table part, not in a cascade segment (cascade segments hold cached
 * keys only).  A bad slot id for it is skipped and flags RC_ERR_DEVICE.
 * Same workspace (attn_decode_workspace) and errors as attn_decode; the latent
 * layout returns RC_ERR_UNSUPPORTED (use kv_store + attn_decode). */
rc_status attn_decode_append(const rc_attn_desc* desc, const void* q, const void* k_new,
                             const void* v_new, const rc_kv_table* kv, int32_t batch,
                             const rc_cascade* cascade, void* out, float* lse, void* ws,
                             size_t ws_bytes, rc_stream_t stream);

/* One decode step of a run handed to attn_decode_steps.  len, max_len: the
 * step's row lengths (device) and their host bound, replacing kv->len and
 * kv->max_len.  store_slots: NULL, or [batch] device slot ids that kv_store
 * fills from k_new/v_new before the step's attention (the latent layout, the
 * FP8 pool).  With store_slots NULL and k_new set the step is an
 * attn_decode_append; with both NULL a plain attn_decode.  ev_begin/ev_end:
 * NULL or a cudaEvent_t recorded on the stream before the step's first launch
 * and after its last (per-step timing). */
typedef struct rc_decode_step {
    const void* q;
    const void* k_new;
    const void* v_new;
    const int32_t* store_slots;
    void* out;
    float* lse;
    const int32_t* len;
    int32_t max_len;
    void* ev_begin;
    void* ev_end;
} rc_decode_step;

/* n_steps decode steps of one batch queued by one call: for step i, in
 * order, its store (if any) and its attn_decode / attn_decode_append, each
 * with the arguments above and the batch's shared table rows, cascade and
 * workspace (sized by attn_decode_workspace for the largest max_len).  Each
 * step computes exactly what the per-step call computes, so the results are
 * those calls' results bit for bit.  One difference in scheduling: when step
 * i and step i-1 are both append steps (k_new given, no store_slots) and no
 * event is recorded between them, step i's cascade kernel reads its q and the
 * cascade segments while step i-1's table pass may still run, and waits for
 * it only before writing its partials (the table pass writes only rows'
 * private last keys).  So every step's q and the segments' keys must be
 * written by work queued before this call, as for any call, and must not be
 * written by it.  The pages describe the
 * decode phase as a loop of one-token steps [LMI decode phase] and a
 * scheduler that keeps the host's work off the GPU's critical path [SGLang
 * engineering article, section 2: the overlap scheduler]; this call takes the
 * per-step host work of that loop down to filling one array.  n_done: NULL or
 * receives the steps queued before the first error (all of them on
 * RC_OK); the first error's status is returned. */
rc_status attn_decode_steps(const rc_attn_desc* desc, const rc_kv_table* kv, int32_t batch,
                            const rc_cascade* cascade, const rc_decode_step* steps, int32_t n_steps,
                            void* ws, size_t ws_bytes, rc_stream_t stream, int32_t* n_done);

/* attn_decode without any device allocation, for callers that cannot call
 * cudaMalloc or hand over a workspace: for example a serving loop whose
 * device memory is all carved up at start-up (the KV pool takes what is left)
 * or a host framework whose plugin interface passes only input and output
 * pointers.  The pages have no counterpart: this is a library convenience.
 * Same arguments, result and errors as attn_decode, minus ws/ws_bytes: the
 * split partials live in a fixed scratch array inside the library,
 * RC_STATIC_SCRATCH_BYTES long, which every GPU that loads the library holds
 * until the process exits.  A call whose partials need more (see
 * attn_decode_workspace) returns RC_ERR_SCRATCH and launches nothing.
 * The first call on a device looks up that device's scratch address (with
 * the device current), so make the first call before any stream capture.
 * The address is kept per device ordinal: it assumes the CUDA runtime's
 * primary context of that device and no cudaDeviceReset afterwards.
 * All calls share the one array, which keeps the last call's contents (the
 * partials are written in full before they are read, so nothing needs
 * clearing): calls that can overlap on the GPU (other streams, other host
 * threads) race on it and must be serialised by the caller. */
#define RC_STATIC_SCRATCH_BYTES (32u << 20)
rc_status attn_decode_static(const rc_attn_desc* desc, const void* q, const rc_kv_table* kv,
                             int32_t batch, const rc_cascade* cascade, void* out, float* lse,
                             rc_stream_t stream);

/* Workspace bytes attn_extend needs (0 today; kept for split variants). */
rc_status attn_extend_workspace(const rc_attn_desc* desc, int32_t batch, int32_t max_q,
                                int32_t max_len, size_t* bytes);

/* Prefill of new tokens over a cached prefix [N49 s.2: only the new part is
 * computed; LMI prefill phase].  Row b has n_b = qo_indptr[b+1]-qo_indptr[b]
 * new tokens, the last n_b positions of its table row (their K/V already
 * stored).  New token i of row b (position p = len[b]-n_b+i) attends to keys
 * 0..p causally.  q and out: [sum n_b][q_heads][head_dim] bf16.
 * max_q: host bound on n_b.  lse: NULL or [sum n_b][q_heads] fp32.
 * Errors: RC_ERR_ARG, RC_ERR_UNSUPPORTED, RC_ERR_CUDA. */
rc_status attn_extend(const rc_attn_desc* desc, const void* q, const int32_t* qo_indptr,
                      const rc_kv_table* kv, int32_t batch, int32_t max_q, void* out,
                      float* lse, void* ws, size_t ws_bytes, rc_stream_t stream);

/* Wait for `stream`, then read and clear the device error word `err` (may be
 * NULL).  A library extra (the pages have no counterpart): it is how errors
 * that kernels detect reach the host, since device calls return at enqueue.  Returns RC_ERR_DEVICE / RC_ERR_TIMEOUT if a kernel flagged one,
 * RC_ERR_CUDA if the stream reported an error, RC_OK otherwise. */
rc_status rc_sync(rc_stream_t stream, int32_t* err);

/* Static string for a status. */
const char* rc_strerror(rc_status status);

/* Self-test of the failure path every kernel's waits share (the pages have no
 * counterpart: this is how a device wait that never completes is reported
 * without faulting the GPU).  Launches one warp on `stream` that waits, with
 * the same bounded mbarrier wait the kernels use, on a barrier nothing ever
 * arrives at; after about a second the wait gives up and the warp ORs the
 * timeout bit into `err` (device int32, caller-owned) and returns, so the
 * context stays usable.  A following rc_sync(stream, err) returns
 * RC_ERR_TIMEOUT and clears the word.  Errors: RC_ERR_ARG (err NULL),
 * RC_ERR_CUDA (launch failed). */
rc_status rc_probe_wait_timeout(int32_t* err, rc_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* RADIXATTN_H */
