// Many query rows over one gathered key list on tcgen05, warp-specialized:
// the kernel body of attn_extend (new tokens over their cached prefix, causal
// among themselves) and of the cascade step of attn_decode (a shared segment
// read once for every request below it).
//
// A CTA owns 256 query rows of one KV head -- two M=128 tiles, each (128/G
// tokens or requests) x (the G query heads of that KV head) -- so every K/V
// tile it gathers feeds both.  Eleven warps with fixed roles:
//   warps 0-3 and 4-7  softmax of query tile 0 and 1: one thread per row /
//                      TMEM lane; read S from TMEM, write P (bf16) back over
//                      it, rescale the row's O in TMEM when its max grows by
//                      more than 2^8;
//   warps 8..8+NP-1    producers, warp 8+i of the tiles t = i mod NP: gather
//                      K/V rows by slot id with 16-byte cp.async into a
//                      5-stage ring (no-swizzle operand layout), each lane's
//                      copies arriving on the stage's mbarrier when they
//                      land;
//   warp 8+NP          issues every MMA (one thread) and owns TMEM.
// Per 64-key tile and query tile q:  S_q = Q_q K^T (M=128, N=64, K=D) into
// one of two S buffers, O_q += P_q V (M=128, N=D, K=64) with P read from
// tensor memory.  The next tile's S products are issued before this tile's
// P.V, so the tensor core works while the softmax warps run, and the softmax
// of tile t+1 does not wait for P.V of tile t (only a rescale of O does).
// TMEM: query tile q uses columns [256q, 256q+256): S buffers at +0 and +64
// (P over their first 32 columns), O at +128.  The tensor core runs one
// thread's MMAs in issue order, so S(t+2) overwrites P(t) only after P(t).V
// has read it.  All hand-offs are mbarriers; every wait is bounded and a wait
// that gives up flags RC_ERR_TIMEOUT.  The MMA thread builds each
// operand's descriptor once and steps it along K with 32-bit adds, and the
// producers' copies of a row carry their offsets as immediates, so neither
// spends issue slots on address arithmetic.
//
// FP8 pool (E4M3 codes, one fp32 scale per (slot, KV head) row): the products
// run in f16 (every E4M3 value is an f16 value; the bf16 queries convert
// exactly within f16's range).  The producers load codes with plain 16-byte
// loads, widen them to f16 in registers and store the operand tiles
// themselves (then fence to the async proxy and arrive), along with the
// tile's 64 K and 64 V scales; the softmax scales S by the K scales and folds
// the V scales into P.  The ring has 4 stages (the scales take the room of
// the fifth).
#pragma once

#include "mq_attn.cuh"
#include "tc.cuh"

namespace rc_tc2 {

constexpr int QT = 2;          // query tiles per CTA
constexpr int TM = 128;        // rows per query tile
constexpr int ROWS = QT * TM;  // query rows per CTA
constexpr int TN = 64;         // keys per tile
constexpr int NS_BF16 = 5;     // K/V stages
constexpr int NS_FP8 = 4;
constexpr int NP = 2;          // producer warps (a third one measured no faster)
constexpr int MMA_WARP = 8 + NP;
constexpr int THREADS = 32 * (MMA_WARP + 1);
constexpr uint32_t kWaitIter = 1u << 24;
template <bool FP8>
__host__ __device__ constexpr int stages() { return FP8 ? NS_FP8 : NS_BF16; }
template <bool FP8>
__host__ __device__ constexpr int n_bars() { return 1 + 2 * stages<FP8>() + 4 + 4 + 2; }

template <int D, bool FP8 = false>
__host__ __device__ constexpr int smem_bytes() {
    return QT * TM * D * 2 + stages<FP8>() * 2 * TN * D * 2 + (FP8 ? stages<FP8>() * 2 * TN * 4 : 0) +
           n_bars<FP8>() * 8 + 16;
}

// The cascade path reads FP8 pools too.
inline constexpr bool fp8_cascade_supported() { return true; }

using tc::ex2;
using tc::fadd2;
using tc::ffma2;
using tc::max3;
using tc::mbar_arrive;

template <int D, int G, rc::MQMode MODE, bool FP8 = false>
__global__ void __launch_bounds__(THREADS, 1) attn_tc2_kernel(const rc::MQParams p) {
    static_assert(!FP8 || D == 128, "FP8 pools: head_dim 128");
    constexpr int NS = stages<FP8>();
    constexpr int kBars = n_bars<FP8>();
    constexpr int CH = D / 8;
    constexpr int TPC = ROWS / G;               // tokens (or requests) per CTA
    constexpr int KV_BYTES = TN * D * 2;
    constexpr uint32_t SB = CH * 128;            // bytes between 8-row groups of Q/K/V tiles
    constexpr uint32_t idS = FP8 ? tc::idesc_f16(TM, TN, false) : tc::idesc_bf16(TM, TN, false);
    constexpr uint32_t idPV = FP8 ? tc::idesc_f16(TM, D, true) : tc::idesc_bf16(TM, D, true);
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* sQ = smem;                                  // [QT][128 rows][D]
    unsigned char* sKV = sQ + QT * TM * D * 2;                 // [NS][K, V]
    float* sScale = reinterpret_cast<float*>(sKV + NS * 2 * KV_BYTES);  // FP8: [NS][K scales, V scales]
    uint64_t* bar = reinterpret_cast<uint64_t*>(sKV + NS * 2 * KV_BYTES + (FP8 ? NS * 2 * TN * 4 : 0));
    uint64_t* q_full = bar + 0;              // count 8 (softmax warps)
    uint64_t* kv_full = bar + 1;             // [NS], count 32 (the lanes of the tile's producer warp)
    uint64_t* kv_empty = bar + 1 + NS;       // [NS], count 1 (MMA commit)
    uint64_t* s_full = bar + 1 + 2 * NS;     // [QT][2], count 1
    uint64_t* p_full = s_full + 4;           // [QT][2] (one per S buffer), count 4 (the tile's softmax warps)
    uint64_t* o_done = p_full + 4;           // [QT], count 1
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + kBars);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = blockIdx.y, z = blockIdx.z;
    int blk = blockIdx.x;
    // cascade: launched as the programmatic dependent of whatever precedes it
    // on the stream (the previous step's table pass), so its CTAs take SMs as
    // that grid drains; nothing is read before that grid has finished.  The
    // table pass of this call is in turn this grid's dependent: it may start
    // once every CTA here has begun (it waits for this grid's end before
    // reading the partials).
    // (early: the wait and the trigger move to just before the first global
    // write, see MQParams::early; the table pass then still launches only
    // after the preceding grid has finished)
    if constexpr (MODE == rc::MQMode::kCascade) {
        if (!p.early) {
            asm volatile("griddepcontrol.wait;\n" ::: "memory");
            asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
        }
    }
    // cascade: this CTA's segment, key chunk and the segment's chunk count.
    // With a compact grid (seg_items > 0) blockIdx.x is the item: one warp
    // walks the segments 32 at a time, each lane counting its segment's
    // (key chunk, row block) items, and a warp scan finds the segment that
    // holds this item (chunk-major inside a segment).
    int c_seg = 0, c_chunk = 0, c_nch = 1;
    if constexpr (MODE == rc::MQMode::kCascade) {
        if (p.seg_items > 0) {
            __shared__ int s_map[4];
            if (threadIdx.x < 32) {
                const int ln = threadIdx.x;
                const int target = blockIdx.x;
                int base = 0, found = -1, f_chunk = 0, f_blk = 0, f_nch = 1;
                for (int s0 = 0; s0 < p.n_seg && found < 0; s0 += 32) {
                    const int sg = s0 + ln;
                    int items = 0, rb = 1, ch = 1;
                    if (sg < p.n_seg) {
                        const int rows = p.seg_row_indptr[sg + 1] - p.seg_row_indptr[sg];
                        const int len = p.seg_indptr[sg + 1] - p.seg_indptr[sg];
                        rb = rows > 0 ? (rows + TPC - 1) / TPC : 1;
                        ch = len > 0 ? min((len + p.seg_chunk - 1) / p.seg_chunk, p.seg_chunks) : 1;
                        items = rows > 0 ? ch * rb : 0;
                    }
                    int incl = items;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const int v = __shfl_up_sync(0xffffffffu, incl, o);
                        if (ln >= o) incl += v;
                    }
                    const int excl = base + incl - items;
                    const unsigned m = __ballot_sync(0xffffffffu, items > 0 && target >= excl && target < excl + items);
                    if (m) {
                        const int src = __ffs(m) - 1;
                        const int j = target - __shfl_sync(0xffffffffu, excl, src);
                        const int rb_s = __shfl_sync(0xffffffffu, rb, src);
                        f_nch = __shfl_sync(0xffffffffu, ch, src);
                        found = s0 + src;
                        f_chunk = j / rb_s;
                        f_blk = j % rb_s;
                    }
                    base += __shfl_sync(0xffffffffu, incl, 31);
                }
                if (ln == 0) {
                    s_map[0] = found;
                    s_map[1] = f_chunk;
                    s_map[2] = f_blk;
                    s_map[3] = f_nch;
                }
            }
            __syncthreads();
            if (s_map[0] < 0) {  // more items than the segments hold: the host arrays differ
                if (threadIdx.x == 0) rc::flag_error(p.err, rc::kErrBadSlot);
                return;
            }
            c_seg = s_map[0];
            c_chunk = s_map[1];
            blk = s_map[2];
            c_nch = s_map[3];
        } else {
            c_seg = z / p.seg_chunks;
            c_chunk = z % p.seg_chunks;
            c_nch = p.seg_chunks;
        }
    }
    const int tok0 = blk * TPC;

    // ---- this CTA's rows and keys (uniform)
    int n_rows_tok, key_count, prefix = 0, qo0, chunk = 0;
    const int32_t* keys;
    if constexpr (MODE == rc::MQMode::kExtend) {
        qo0 = p.qo_indptr[z];
        n_rows_tok = p.qo_indptr[z + 1] - qo0;
        const int L = p.len[z];
        prefix = L - n_rows_tok;
        const int64_t row0 = p.start[z];
        if (tok0 >= n_rows_tok) return;
        if (row0 < 0 || prefix < 0 || row0 + L > p.table_len) {
            if (tid == 0) rc::flag_error(p.err, rc::kErrBadSlot);
            return;
        }
        keys = p.table + row0;
        key_count = prefix + min(n_rows_tok, tok0 + TPC);
    } else {
        const int seg = c_seg;
        chunk = c_chunk;
        qo0 = p.seg_row_indptr[seg];
        n_rows_tok = p.seg_row_indptr[seg + 1] - qo0;
        const int k0 = chunk * p.seg_chunk;
        keys = p.seg_slots + p.seg_indptr[seg] + k0;
        key_count = min(p.seg_indptr[seg + 1] - p.seg_indptr[seg] - k0, p.seg_chunk);
        if (tok0 >= n_rows_tok) return;
        // compact grid: no CTA runs past the segment's last chunk, so its
        // first chunk's CTA marks those partials empty for its rows
        if (p.seg_items > 0 && !p.early && chunk == 0 && c_nch < p.seg_chunks && tid < ROWS) {
            const int tk = tok0 + tid / G;
            if (tk < n_rows_tok)
                for (int c = c_nch; c < p.seg_chunks; ++c)
                    p.part_lse[((int64_t)(qo0 + tk) * p.q_heads + kvh * G + (tid % G)) * p.seg_chunks + c] = -INFINITY;
        }
        if (key_count <= 0) {  // segment shorter than this chunk: an empty partial
            if (p.early) {
                asm volatile("griddepcontrol.wait;\n" ::: "memory");
                asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
                if (p.seg_items > 0 && chunk == 0 && tid < ROWS) {
                    const int tk = tok0 + tid / G;
                    if (tk < n_rows_tok)
                        for (int c = c_nch; c < p.seg_chunks; ++c)
                            p.part_lse[((int64_t)(qo0 + tk) * p.q_heads + kvh * G + (tid % G)) * p.seg_chunks + c] =
                                -INFINITY;
                }
            }
            if (tid < ROWS) {
                const int tk = tok0 + tid / G;
                if (tk < n_rows_tok)
                    p.part_lse[((int64_t)(qo0 + tk) * p.q_heads + kvh * G + (tid % G)) * p.seg_chunks + chunk] =
                        -INFINITY;
            }
            return;
        }
    }
    // a wait gave up in an earlier CTA: the results are void, leave at once,
    // all threads alike (the word can change between two threads' reads, and
    // a CTA split here would stall at its first barrier)
    if (__syncthreads_or(p.err && (*reinterpret_cast<volatile int32_t*>(p.err) & rc::kErrTimeout))) return;
    const int n_tiles = (key_count + TN - 1) / TN;
    // query tiles with at least one valid row
    const int n_qt = min(QT, ((min(n_rows_tok - tok0, TPC) * G) + TM - 1) / TM);

    // producers: slot ids of their first tile, loaded before the set-up too
    int sl_first[2] = {-1, -1};
    if (warp >= 8 && warp < MMA_WARP) {
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int key = (warp - 8) * TN + lane + 32 * h2;
            if (warp - 8 < n_tiles && key < key_count) sl_first[h2] = __ldg(keys + key);
        }
    }
    if (warp < 8) {
        // Q rows of query tile warp/4, issued first so that their latency
        // overlaps the set-up.  The row indices (cascade: a gather through
        // seg_rows) are all loaded before the first copy is issued.
        const int q = warp >> 2, r = tid & 127;
        unsigned char* sQq = sQ + q * TM * D * 2;
        int64_t qrow[CH];
        bool qok[CH];
#pragma unroll
        for (int i = 0; i < CH; ++i) {
            const int gi = r + 128 * i;
            const int rr = (gi & 7) + 8 * (gi / (8 * CH));
            const int qr = q * TM + rr;
            const int tk = tok0 + qr / G;
            const int h = kvh * G + (qr % G);
            qok[i] = tk < n_rows_tok;
            if constexpr (MODE == rc::MQMode::kExtend) qrow[i] = (int64_t)(qo0 + tk) * p.q_heads + h;
            else qrow[i] = qok[i] ? (int64_t)__ldg(p.seg_rows + qo0 + tk) * p.q_heads + h : 0;
            if (!qok[i]) qrow[i] = 0;
        }
        if constexpr (FP8) {  // f16 operand: load, convert, store
            uint4 qv[CH];
#pragma unroll
            for (int i = 0; i < CH; ++i) {
                const int c = ((r + 128 * i) >> 3) % CH;
                qv[i] = qok[i] ? __ldg(reinterpret_cast<const uint4*>(p.q + qrow[i] * D + c * 8)) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < CH; ++i) {
                const int gi = r + 128 * i;
                const int rr = (gi & 7) + 8 * (gi / (8 * CH));
                const int c = (gi >> 3) % CH;
                *reinterpret_cast<uint4*>(sQq + tc::cm_offset(rr, c, CH)) =
                    make_uint4(rc::bf16x2_to_f16x2(qv[i].x), rc::bf16x2_to_f16x2(qv[i].y),
                               rc::bf16x2_to_f16x2(qv[i].z), rc::bf16x2_to_f16x2(qv[i].w));
            }
        } else {
#pragma unroll
            for (int i = 0; i < CH; ++i) {
                const int gi = r + 128 * i;
                const int rr = (gi & 7) + 8 * (gi / (8 * CH));
                const int c = (gi >> 3) % CH;
                rc::cp_async16(rc::smem_u32(sQq + tc::cm_offset(rr, c, CH)), p.q + qrow[i] * D + c * 8,
                               qok[i] ? 16u : 0u);
            }
            rc::cp_async_commit();
        }
    }
    if (tid == 0) {
        tc::mbar_init(q_full, 8);
        for (int s = 0; s < NS; ++s) {
            tc::mbar_init(&kv_full[s], 32);
            tc::mbar_init(&kv_empty[s], 1);
        }
        for (int i = 0; i < 4; ++i) {
            tc::mbar_init(&s_full[i], 1);
            tc::mbar_init(&p_full[i], 4);
        }
        for (int q = 0; q < QT; ++q) {
            tc::mbar_init(&o_done[q], 1);
        }
        tc::fence_mbar_init();
    }
    if (warp == MMA_WARP) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tbase = *tslot;
    bool ok = true;

    if (warp < 8) {
        // ================================================= softmax warpgroups
        const int q = warp >> 2;             // query tile
        const int r = tid & 127;             // row within the tile = TMEM lane
        const int row = q * TM + r;          // row within the CTA
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const uint32_t tq = tbase + q * 256 + lane_off;
        rc::cp_async_wait<0>();  // this thread's Q chunks (issued before the set-up)
        tc::fence_proxy_async();
        __syncwarp();
        if (lane == 0) mbar_arrive(q_full);

        const int r_tok = tok0 + row / G;
        const bool row_valid = r_tok < n_rows_tok;
        int lim;
        if constexpr (MODE == rc::MQMode::kExtend) lim = row_valid ? prefix + r_tok + 1 : 0;
        else lim = row_valid ? key_count : 0;
        const float sc = p.scale_log2;
        float m_used = -INFINITY, l_run = 0.f;
        if (q < n_qt) {
            for (int t = 0; t < n_tiles && ok; ++t) {
                ok = __all_sync(0xffffffffu, tc::mbar_wait(&s_full[q * 2 + (t & 1)], (t >> 1) & 1, kWaitIter));
                tc::fence_after();
                const uint32_t tS = tq + (t & 1) * TN;
                uint32_t sa[32], sb[32];
                tc::tmem_ld32_issue(tS, sa);
                tc::tmem_ld32_issue(tS + 32, sb);
                tc::tmem_ld_wait(sa);
                tc::tmem_ld_wait(sb);
                float s[TN];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    s[j] = __uint_as_float(sa[j]);
                    s[32 + j] = __uint_as_float(sb[j]);
                }
                const float* tsc = sScale + (t % NS) * 2 * TN;  // FP8: this tile's K then V scales
                if constexpr (FP8) {
                    // the producer's scale stores are visible once its arrival
                    // on the stage is (that phase completed before S(t) ran)
                    ok = __all_sync(0xffffffffu, tc::mbar_wait(&kv_full[t % NS], (t / NS) & 1, kWaitIter)) && ok;
#pragma unroll
                    for (int j = 0; j < TN; ++j) s[j] *= tsc[j];
                }
                const int kb = t * TN;
                if (kb + TN > lim) {  // the causal edge or the end of the keys
#pragma unroll
                    for (int j = 0; j < TN; ++j)
                        if (kb + j >= lim) s[j] = -INFINITY;
                }
                float m8[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    m8[i] = max3(s[i], s[8 + i], s[16 + i]);
                    m8[i] = max3(m8[i], s[24 + i], s[32 + i]);
                    m8[i] = max3(m8[i], s[40 + i], s[48 + i]);
                    m8[i] = fmaxf(m8[i], s[56 + i]);
                }
                const float mraw = max3(max3(m8[0], m8[1], m8[2]), max3(m8[3], m8[4], m8[5]), fmaxf(m8[6], m8[7]));
                const float mt = mraw * sc;  // sc > 0: the max of the scaled row
                const bool grow = mt > m_used + 8.f;
                const bool rescale_o = grow && m_used != -INFINITY;
                if (__any_sync(0xffffffffu, rescale_o)) {
                    // O must be stable: the previous tile's P.V has completed
                    ok = __all_sync(0xffffffffu, tc::mbar_wait(&o_done[q], (t - 1) & 1, kWaitIter)) && ok;
                    tc::fence_after();
                    const float a = rescale_o ? ex2(m_used - mt) : 1.f;
#pragma unroll
                    for (int c = 0; c < D / 32; ++c) {
                        uint32_t v[32];
                        tc::tmem_ld32_issue(tq + 128 + c * 32, v);
                        tc::tmem_ld_wait(v);
#pragma unroll
                        for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * a);
                        tc::tmem_st32_issue(tq + 128 + c * 32, v);
                    }
                    tc::tmem_st_wait();
                }
                if (grow) {
                    l_run *= ex2(m_used - mt);  // 0 while nothing was seen
                    m_used = mt;
                }
                const float nmu = m_used == -INFINITY ? 0.f : -m_used;
                uint32_t pk[32];
                float2 ls[4] = {{0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float2 x = ffma2(make_float2(s[2 * i], s[2 * i + 1]), sc, nmu);
                    const float2 e = make_float2(ex2(x.x), ex2(x.y));
                    ls[i & 3] = fadd2(ls[i & 3], e);
                    if constexpr (FP8) pk[i] = rc::pack_f16(e.x * tsc[TN + 2 * i], e.y * tsc[TN + 2 * i + 1]);
                    else pk[i] = rc::pack_bf16(e.x, e.y);
                }
                // P (bf16) over the first half of this S buffer: the A operand of P.V
                tc::tmem_st32_issue(tS, pk);
                const float2 l01 = fadd2(fadd2(ls[0], ls[1]), fadd2(ls[2], ls[3]));
                l_run += l01.x + l01.y;
                tc::tmem_st_wait();
                // Last tile: see P(n-2).V done before handing over P(n-1), while
                // o_done can only be at phase n-2 or n-1 (a parity wait tells
                // two phases apart, not three; S(n-1) guarantees P(n-3).V).
                if (t == n_tiles - 1 && t > 0) {
                    ok = __all_sync(0xffffffffu, tc::mbar_wait(&o_done[q], (t - 1) & 1, kWaitIter)) && ok;
                    tc::fence_after();
                }
                tc::fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[q * 2 + (t & 1)]);
            }
            // the last P.V: o_done is at phase n-1 or n here
            if (ok && n_tiles > 0)
                ok = __all_sync(0xffffffffu, tc::mbar_wait(&o_done[q], (n_tiles - 1) & 1, kWaitIter));
            tc::fence_after();
        }
        if (!ok) rc::flag_error(p.err, rc::kErrTimeout);
        if constexpr (MODE == rc::MQMode::kCascade) {
            if (p.early) {  // the partials below are what the preceding grid read
                asm volatile("griddepcontrol.wait;\n" ::: "memory");
                asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
                if (p.seg_items > 0 && chunk == 0 && c_nch < p.seg_chunks) {
                    const int tk = tok0 + tid / G;  // tid < ROWS here
                    if (tk < n_rows_tok)
                        for (int c = c_nch; c < p.seg_chunks; ++c)
                            p.part_lse[((int64_t)(qo0 + tk) * p.q_heads + kvh * G + (tid % G)) * p.seg_chunks + c] =
                                -INFINITY;
                }
            }
        }
        // ---- epilogue: normalised O rows and their log-sum-exp.  Rows go out
        // through shared memory so that each store instruction writes whole
        // row segments: per 32 columns, the warp's 32x32 fp32 block is staged
        // (16-byte chunks XOR-swizzled by row: conflict-free both ways) in
        // this warp's 4 KB of the Q region -- free once the tile's last P.V
        // is done, since every S product was issued before it -- and read
        // back 8 lanes per row, 4 rows per instruction.
        if (q < n_qt) {
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            const float lse2 = l_run > 0.f ? m_used + log2f(l_run) : -INFINITY;
            float* stg = reinterpret_cast<float*>(sQ + warp * 4096);
            const int k8 = lane & 7;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {
                uint32_t vb[32];
                tc::tmem_ld32_issue(tq + 128 + c * 32, vb);
                tc::tmem_ld_wait(vb);
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    *reinterpret_cast<float4*>(stg + lane * 32 + ((k ^ (lane & 7)) * 4)) =
                        make_float4(__uint_as_float(vb[4 * k]) * inv, __uint_as_float(vb[4 * k + 1]) * inv,
                                    __uint_as_float(vb[4 * k + 2]) * inv, __uint_as_float(vb[4 * k + 3]) * inv);
                __syncwarp();
#pragma unroll
                for (int pass = 0; pass < 8; ++pass) {
                    const int rr = pass * 4 + (lane >> 3);
                    const float4 f = *reinterpret_cast<const float4*>(stg + rr * 32 + ((k8 ^ (rr & 7)) * 4));
                    const int rc_ = q * TM + (warp & 3) * 32 + rr;  // row within the CTA
                    const int tk = tok0 + rc_ / G;
                    const int hh = kvh * G + (rc_ % G);
                    if (!ok || tk >= n_rows_tok) continue;
                    if constexpr (MODE == rc::MQMode::kExtend) {
                        uint2 w;
                        w.x = rc::pack_bf16(f.x, f.y);
                        w.y = rc::pack_bf16(f.z, f.w);
                        *reinterpret_cast<uint2*>(p.out + ((int64_t)(qo0 + tk) * p.q_heads + hh) * D + c * 32 + k8 * 4) =
                            w;
                    } else {
                        *reinterpret_cast<float4*>(
                            p.part_o + (((int64_t)(qo0 + tk) * p.q_heads + hh) * p.seg_chunks + chunk) * D + c * 32 +
                            k8 * 4) = f;
                    }
                }
                __syncwarp();
            }
            if (ok && row_valid) {
                const int h = kvh * G + (row % G);
                if constexpr (MODE == rc::MQMode::kExtend) {
                    if (p.lse) p.lse[(int64_t)(qo0 + r_tok) * p.q_heads + h] = lse2 * rc::kLn2;
                } else {
                    p.part_lse[((int64_t)(qo0 + r_tok) * p.q_heads + h) * p.seg_chunks + chunk] = lse2;
                }
            }
        }
    } else if (warp < MMA_WARP) {
        // ============================================== producers (NP warps)
        // warp 8+i loads the tiles t = i mod NP, each as far ahead as free
        // stages allow (completion is signalled on the stage's barrier by the
        // copies themselves), reading the slot ids of its next tile one tile
        // ahead.
        // lane -> (key within an 8-key group, 16-byte column within a group of 4)
        const int klo = lane & 7, csub = lane >> 3;
        // keys here are shared: by the CTAs of the other row blocks, and (a
        // cached prefix) by later steps -- keep them in L2
        const uint64_t pol = rc::l2_policy_evict_last();
        const int t0 = warp - 8;
        auto load_ids = [&](int t, int (&sl)[2]) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int key = t * TN + lane + 32 * h2;
                sl[h2] = (t < n_tiles && key < key_count) ? __ldg(keys + key) : -1;
            }
        };
        int sl[2] = {sl_first[0], sl_first[1]}, sl_next[2];
        for (int t = t0; t < n_tiles && ok; t += NP) {
            const int s = t % NS;
            load_ids(t + NP, sl_next);
            if (t >= NS) ok = __all_sync(0xffffffffu, tc::mbar_wait(&kv_empty[s], ((t / NS) + 1) & 1, kWaitIter));
            if (!ok) break;
            unsigned char* sK = sKV + s * 2 * KV_BYTES;
            unsigned char* sV = sK + KV_BYTES;
            if constexpr (FP8) {
                // 16 E4M3 codes per load (8 keys x 64 bytes per instruction,
                // so the 16-byte f16 stores of 8 keys are 128 contiguous bytes);
                // the K and V loads of the tile are all in flight together
                uint4 w2[2][TN / 8][2];
#pragma unroll
                for (int kg = 0; kg < TN / 8; ++kg) {
                    const int key = kg * 8 + klo;
                    int slot = __shfl_sync(0xffffffffu, sl[kg >> 2], (kg & 3) * 8 + klo);
                    bool live = t * TN + key < key_count;
                    if (live && (slot < 0 || (int64_t)slot >= p.n_slots)) {
                        rc::flag_error(p.err, rc::kErrBadSlot);
                        live = false;
                    }
                    const int64_t base = ((int64_t)(live ? slot : 0) * p.kv_heads + kvh) * D;
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        const unsigned char* src = reinterpret_cast<const unsigned char*>(m ? p.pool_v : p.pool_k);
#pragma unroll
                        for (int cg = 0; cg < 2; ++cg)
                            w2[m][kg][cg] = live ? __ldg(reinterpret_cast<const uint4*>(src + base + (cg * 4 + csub) * 16))
                                                 : make_uint4(0, 0, 0, 0);
                    }
                }
#pragma unroll
                for (int m = 0; m < 2; ++m) {
                    unsigned char* dst = m ? sV : sK;
                    auto& w = w2[m];
#pragma unroll
                    for (int kg = 0; kg < TN / 8; ++kg) {
                        const int key = kg * 8 + klo;
#pragma unroll
                        for (int cg = 0; cg < 2; ++cg) {
                            const int c8 = cg * 4 + csub;  // 16-code chunk: f16 chunks 2*c8, 2*c8+1
                            const uint4 x = w[kg][cg];
                            uint4 f0, f1;
                            rc::e4m3x4_to_f16x4(x.x, f0.x, f0.y);
                            rc::e4m3x4_to_f16x4(x.y, f0.z, f0.w);
                            rc::e4m3x4_to_f16x4(x.z, f1.x, f1.y);
                            rc::e4m3x4_to_f16x4(x.w, f1.z, f1.w);
                            *reinterpret_cast<uint4*>(dst + tc::cm_offset(key, 2 * c8, CH)) = f0;
                            *reinterpret_cast<uint4*>(dst + tc::cm_offset(key, 2 * c8 + 1, CH)) = f1;
                        }
                    }
                }
                float* tsc = sScale + s * 2 * TN;
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int key = lane + 32 * h2;
                    const int slot = sl[h2];
                    const bool live = t * TN + key < key_count && slot >= 0 && (int64_t)slot < p.n_slots;
                    const int64_t row = (int64_t)(live ? slot : 0) * p.kv_heads + kvh;
                    tsc[key] = live ? __ldg(p.k_scale + row) : 0.f;
                    tsc[TN + key] = live ? __ldg(p.v_scale + row) : 0.f;
                }
                tc::fence_proxy_async();  // this lane's stores, before the tensor core reads them
                mbar_arrive(&kv_full[s]);
                sl[0] = sl_next[0];
                sl[1] = sl_next[1];
                continue;
            }
#pragma unroll
            for (int kg = 0; kg < TN / 8; ++kg) {
                const int key = kg * 8 + klo;
                int slot = __shfl_sync(0xffffffffu, sl[kg >> 2], (kg & 3) * 8 + klo);
                uint32_t bytes = 16;
                if (t * TN + key >= key_count) { slot = 0; bytes = 0; }
                else if (slot < 0 || (int64_t)slot >= p.n_slots) {
                    rc::flag_error(p.err, rc::kErrBadSlot);
                    slot = 0;
                    bytes = 0;
                }
                // chunks c = 4 cg + csub: 512 bytes apart in the stage, 64 in the row
                const int64_t base = ((int64_t)slot * p.kv_heads + kvh) * D + csub * 8;
                const uint32_t off = tc::cm_offset(key, csub, CH);
                rc::cp_async16_run<512, 64>(rc::smem_u32(sK) + off, p.pool_k + base, bytes, pol,
                                            std::make_integer_sequence<int, CH / 4>{});
                rc::cp_async16_run<512, 64>(rc::smem_u32(sV) + off, p.pool_v + base, bytes, pol,
                                            std::make_integer_sequence<int, CH / 4>{});
            }
            // each lane arrives on the stage's barrier when its copies have
            // landed; the warp goes on to the next tile at once
            tc::cp_async_mbar_arrive(&kv_full[s]);
            sl[0] = sl_next[0];
            sl[1] = sl_next[1];
        }
        rc::cp_async_wait<0>();  // nothing in flight when the warp leaves
        if (!ok) rc::flag_error(p.err, rc::kErrTimeout);
    } else if (lane == 0) {
        // ================================================= MMA (warp 8+NP)
        // descriptors built once per operand and stepped along K by 32-bit adds
        const tc::Desc qd = tc::desc_halves(rc::smem_u32(sQ), 128, SB);
        auto issue_s = [&](int t) {
            const tc::Desc kd = tc::desc_halves(rc::smem_u32(sKV + (t % NS) * 2 * KV_BYTES), 128, SB);
            for (int q = 0; q < n_qt; ++q) {
                const uint32_t qlo = qd.lo + q * (TM * D * 2 / 16);
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    tc::mma_bf16_h(tbase + q * 256 + (t & 1) * TN, qlo + k * 16, qd.hi, kd.lo + k * 16, kd.hi, idS,
                                   k > 0 ? 1u : 0u);
                tc::commit(&s_full[q * 2 + (t & 1)]);
            }
        };
        ok = tc::mbar_wait(q_full, 0, kWaitIter);
        if (ok && n_tiles > 0) {
            ok = tc::mbar_wait(&kv_full[0], 0, kWaitIter);
            tc::fence_after();
            tc::fence_proxy_async();  // the rows arrived through the generic proxy; the tensor core reads them
            if (ok) issue_s(0);
        }
        for (int t = 0; t < n_tiles && ok; ++t) {
            const int s = t % NS;
            if (t + 1 < n_tiles) {  // next tile's S products first: they run during this softmax
                ok = tc::mbar_wait(&kv_full[(t + 1) % NS], ((t + 1) / NS) & 1, kWaitIter);
                tc::fence_after();
                tc::fence_proxy_async();
                if (!ok) break;
                issue_s(t + 1);
            }
            const tc::Desc vd = tc::desc_halves(rc::smem_u32(sKV + s * 2 * KV_BYTES + KV_BYTES), SB, 128);
            for (int q = 0; q < n_qt && ok; ++q) {
                ok = tc::mbar_wait(&p_full[q * 2 + (t & 1)], (t >> 1) & 1, kWaitIter);
                tc::fence_after();
                if (!ok) break;
                const uint32_t pt = tbase + q * 256 + (t & 1) * TN;  // P(t) in TMEM, 8 columns per 16 keys
#pragma unroll
                for (int j = 0; j < TN / 16; ++j)
                    tc::mma_bf16_ts_h(tbase + q * 256 + 128, pt + j * 8, vd.lo + j * (2 * SB / 16), vd.hi, idPV,
                                      (t > 0 || j > 0) ? 1u : 0u);
                tc::commit(&o_done[q]);
            }
            tc::commit(&kv_empty[s]);  // stage s is free once everything issued so far is done
        }
        if (!ok) rc::flag_error(p.err, rc::kErrTimeout);
    }
    if constexpr (MODE == rc::MQMode::kCascade) {
        if (p.early) {  // every thread of the CTA has waited and triggered before it leaves
            asm volatile("griddepcontrol.wait;\n" ::: "memory");
            asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == MMA_WARP) {
        tc::fence_after();
        tc::tmem_dealloc(tbase, 512);
    }
}

}  // namespace rc_tc2
