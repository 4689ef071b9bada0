// Many query rows over one gathered key list on tcgen05, warp-specialized:
// the kernel body of attn_extend (new tokens over their cached prefix, causal
// among themselves) and of the cascade step of attn_decode (a shared segment
// read once for every request below it).
//
// A CTA owns 256 query rows of one KV head -- two M=128 tiles, each (128/G
// tokens or requests) x (the G query heads of that KV head) -- so every K/V
// tile it gathers feeds both.  Eleven warps with fixed roles:
//   warps 0-3 and 4-7  softmax of query tile 0 and 1: one thread per row /
//                      TMEM lane; read S, write P (bf16) to shared memory,
//                      rescale the row's O in TMEM when its max grows > 2^8;
//   warps 8, 9         producers of the even and odd tiles: gather K/V rows
//                      by slot id with cp.async into a 4-stage ring
//                      (no-swizzle operand layout);
//   warp 10            issues every MMA (one thread) and owns TMEM.
// Per 64-key tile and query tile q:  S_q = Q_q K^T (M=128, N=64, K=D) into
// one of two S buffers, O_q += P_q V (M=128, N=D, K=64).  The next tile's S
// products are issued before this tile's P.V, so the tensor core works while
// the softmax warps run.  TMEM: query tile q uses columns [256q, 256q+256):
// S buffers at +0 and +64, O at +128.  All hand-offs are mbarriers; every
// wait is bounded and a wait that gives up flags RC_ERR_TIMEOUT.
#pragma once

#include "mq_attn.cuh"
#include "tc.cuh"

namespace rc_tc2 {

constexpr int QT = 2;          // query tiles per CTA
constexpr int TM = 128;        // rows per query tile
constexpr int ROWS = QT * TM;  // query rows per CTA
constexpr int TN = 64;         // keys per tile
constexpr int NS = 4;          // K/V stages
constexpr int THREADS = 352;
constexpr uint32_t kWaitIter = 1u << 24;

template <int D>
__host__ __device__ constexpr int smem_bytes() {
    return QT * TM * D * 2 + NS * 2 * TN * D * 2 + QT * TM * TN * 2 + 18 * 8 + 16;
}

RC_DEV void mbar_arrive(uint64_t* mbar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}\n" ::"r"(rc::smem_u32(mbar))
                 : "memory");
}

template <int D, int G, rc::MQMode MODE>
__global__ void __launch_bounds__(THREADS, 1) attn_tc2_kernel(const rc::MQParams p) {
    constexpr int CH = D / 8;
    constexpr int TPC = ROWS / G;               // tokens (or requests) per CTA
    constexpr int KV_BYTES = TN * D * 2;
    constexpr uint32_t SB = CH * 128;            // bytes between 8-row groups of Q/K/V tiles
    constexpr uint32_t idS = tc::idesc_bf16(TM, TN, false);
    constexpr uint32_t idPV = tc::idesc_bf16(TM, D, true);
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* sQ = smem;                                  // [QT][128 rows][D]
    unsigned char* sKV = sQ + QT * TM * D * 2;                 // [NS][K, V]
    unsigned char* sP = sKV + NS * 2 * KV_BYTES;               // [QT][128 rows][64 keys]
    uint64_t* bar = reinterpret_cast<uint64_t*>(sP + QT * TM * TN * 2);
    uint64_t* q_full = bar + 0;          // count 256 (softmax threads)
    uint64_t* kv_full = bar + 1;         // [NS], count 32 (the lanes of the tile's producer warp)
    uint64_t* kv_empty = bar + 5;        // [NS], count 1 (MMA commit)
    uint64_t* s_full = bar + 9;          // [QT][2], count 1
    uint64_t* p_full = bar + 13;         // [QT], count 128
    uint64_t* o_done = bar + 15;         // [QT], count 1
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 18);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = blockIdx.y, z = blockIdx.z, blk = blockIdx.x;
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
        const int seg = z / p.seg_chunks;
        chunk = z % p.seg_chunks;
        qo0 = p.seg_row_indptr[seg];
        n_rows_tok = p.seg_row_indptr[seg + 1] - qo0;
        const int k0 = chunk * p.seg_chunk;
        keys = p.seg_slots + p.seg_indptr[seg] + k0;
        key_count = min(p.seg_indptr[seg + 1] - p.seg_indptr[seg] - k0, p.seg_chunk);
        if (tok0 >= n_rows_tok) return;
        if (key_count <= 0) {  // segment shorter than this chunk: an empty partial
            if (tid < ROWS) {
                const int tk = tok0 + tid / G;
                if (tk < n_rows_tok)
                    p.part_lse[((int64_t)(qo0 + tk) * p.q_heads + kvh * G + (tid % G)) * p.seg_chunks + chunk] =
                        -INFINITY;
            }
            return;
        }
    }
    const int n_tiles = (key_count + TN - 1) / TN;
    // query tiles with at least one valid row
    const int n_qt = min(QT, ((min(n_rows_tok - tok0, TPC) * G) + TM - 1) / TM);

    if (tid == 0) {
        tc::mbar_init(q_full, QT * TM);
        for (int s = 0; s < NS; ++s) {
            tc::mbar_init(&kv_full[s], 32);
            tc::mbar_init(&kv_empty[s], 1);
        }
        for (int i = 0; i < 4; ++i) tc::mbar_init(&s_full[i], 1);
        for (int q = 0; q < QT; ++q) {
            tc::mbar_init(&p_full[q], TM);
            tc::mbar_init(&o_done[q], 1);
        }
        tc::fence_mbar_init();
    }
    if (warp == 10) {
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
        unsigned char* sQq = sQ + q * TM * D * 2;
        unsigned char* sPq = sP + q * TM * TN * 2;
        // Q rows of this tile (zero past the end)
        for (int gi = r; gi < TM * CH; gi += 128) {
            const int rr = (gi & 7) + 8 * (gi / (8 * CH));
            const int c = (gi >> 3) % CH;
            const int qr = q * TM + rr;
            const int tk = tok0 + qr / G;
            const int h = kvh * G + (qr % G);
            int64_t qrow = 0;
            if (tk < n_rows_tok) {
                if constexpr (MODE == rc::MQMode::kExtend) qrow = (int64_t)(qo0 + tk) * p.q_heads + h;
                else qrow = (int64_t)p.seg_rows[qo0 + tk] * p.q_heads + h;
            }
            rc::cp_async16(rc::smem_u32(sQq + tc::cm_offset(rr, c, CH)), p.q + qrow * D + c * 8,
                           tk < n_rows_tok ? 16u : 0u);
        }
        rc::cp_async_commit();
        rc::cp_async_wait<0>();
        tc::fence_proxy_async();
        mbar_arrive(q_full);

        const int r_tok = tok0 + row / G;
        const bool row_valid = r_tok < n_rows_tok;
        int lim;
        if constexpr (MODE == rc::MQMode::kExtend) lim = row_valid ? prefix + r_tok + 1 : 0;
        else lim = row_valid ? key_count : 0;
        float m_used = -INFINITY, l_run = 0.f;
        if (q < n_qt) {
            for (int t = 0; t < n_tiles && ok; ++t) {
                ok = __all_sync(0xffffffffu, tc::mbar_wait(&s_full[q * 2 + (t & 1)], (t >> 1) & 1, kWaitIter));
                tc::fence_after();
                float s[TN];
                const uint32_t tS = tq + (t & 1) * TN;
                tc::tmem_ld32(tS, *reinterpret_cast<float(*)[32]>(&s[0]));
                tc::tmem_ld32(tS + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
                const int kb = t * TN;
                float mt = -INFINITY;
#pragma unroll
                for (int j = 0; j < TN; ++j) {
                    s[j] = kb + j < lim ? s[j] * p.scale_log2 : -INFINITY;
                    mt = fmaxf(mt, s[j]);
                }
                // P.V of the previous tile must be done: O stable, P buffer free
                if (t > 0) {
                    ok = __all_sync(0xffffffffu, tc::mbar_wait(&o_done[q], (t - 1) & 1, kWaitIter)) && ok;
                    tc::fence_after();
                }
                if (mt > m_used + 8.f) {
                    if (t > 0 && m_used != -INFINITY) {
                        const float a = rc::fast_exp2(m_used - mt);
#pragma unroll
                        for (int c = 0; c < D / 32; ++c) {
                            float v[32];
                            tc::tmem_ld32(tq + 128 + c * 32, v);
#pragma unroll
                            for (int j = 0; j < 32; ++j) v[j] *= a;
                            tc::tmem_st32(tq + 128 + c * 32, v);
                        }
                        l_run *= a;
                    }
                    m_used = mt;
                }
                const float mu = m_used == -INFINITY ? 0.f : m_used;
#pragma unroll
                for (int c = 0; c < TN / 8; ++c) {
                    float e[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        e[j] = rc::fast_exp2(s[c * 8 + j] - mu);
                        l_run += e[j];
                    }
                    uint4 w;
                    w.x = rc::pack_bf16(e[0], e[1]);
                    w.y = rc::pack_bf16(e[2], e[3]);
                    w.z = rc::pack_bf16(e[4], e[5]);
                    w.w = rc::pack_bf16(e[6], e[7]);
                    *reinterpret_cast<uint4*>(sPq + tc::cm_offset(r, c, TN / 8)) = w;
                }
                tc::fence_proxy_async();
                tc::fence_before();
                mbar_arrive(&p_full[q]);
            }
            if (ok && n_tiles > 0)
                ok = __all_sync(0xffffffffu, tc::mbar_wait(&o_done[q], (n_tiles - 1) & 1, kWaitIter));
            tc::fence_after();
        }
        if (!ok) rc::flag_error(p.err, rc::kErrTimeout);
        // ---- epilogue: normalised O row (and its log-sum-exp)
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const float lse2 = l_run > 0.f ? m_used + log2f(l_run) : -INFINITY;
        const bool write = ok && row_valid && q < n_qt;
        const int h = kvh * G + (row % G);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            float v[32];
            tc::tmem_ld32(tq + 128 + c * 32, v);
            if (!write) continue;
            if constexpr (MODE == rc::MQMode::kExtend) {
                __nv_bfloat16* dst = p.out + ((int64_t)(qo0 + r_tok) * p.q_heads + h) * D + c * 32;
#pragma unroll
                for (int j = 0; j < 32; j += 8) {
                    uint4 w;
                    w.x = rc::pack_bf16(v[j] * inv, v[j + 1] * inv);
                    w.y = rc::pack_bf16(v[j + 2] * inv, v[j + 3] * inv);
                    w.z = rc::pack_bf16(v[j + 4] * inv, v[j + 5] * inv);
                    w.w = rc::pack_bf16(v[j + 6] * inv, v[j + 7] * inv);
                    *reinterpret_cast<uint4*>(dst + j) = w;
                }
            } else {
                float* dst =
                    p.part_o + (((int64_t)(qo0 + r_tok) * p.q_heads + h) * p.seg_chunks + chunk) * D + c * 32;
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4*>(dst + j) =
                        make_float4(v[j] * inv, v[j + 1] * inv, v[j + 2] * inv, v[j + 3] * inv);
            }
        }
        if (write) {
            if constexpr (MODE == rc::MQMode::kExtend) {
                if (p.lse) p.lse[(int64_t)(qo0 + r_tok) * p.q_heads + h] = lse2 * rc::kLn2;
            } else {
                p.part_lse[((int64_t)(qo0 + r_tok) * p.q_heads + h) * p.seg_chunks + chunk] = lse2;
            }
        }
    } else if (warp == 8 || warp == 9) {
        // ============================================== producers (2 warps)
        // warp 8 loads the even tiles, warp 9 the odd ones; each keeps one of
        // its tiles in flight while it issues the next, and reads the slot ids
        // of its next tile one tile ahead.
        // lane -> (key within an 8-key group, 16-byte column within a group of 4)
        const int klo = lane & 7, csub = lane >> 3;
        const int t0 = warp - 8;
        auto load_ids = [&](int t, int (&sl)[2]) {
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                const int key = t * TN + lane + 32 * h2;
                sl[h2] = (t < n_tiles && key < key_count) ? __ldg(keys + key) : -1;
            }
        };
        int sl[2], sl_next[2];
        load_ids(t0, sl);
        int prev = -1;
        for (int t = t0; t < n_tiles && ok; t += 2) {
            const int s = t % NS;
            load_ids(t + 2, sl_next);
            if (t >= NS) ok = __all_sync(0xffffffffu, tc::mbar_wait(&kv_empty[s], ((t / NS) + 1) & 1, kWaitIter));
            if (!ok) break;
            unsigned char* sK = sKV + s * 2 * KV_BYTES;
            unsigned char* sV = sK + KV_BYTES;
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
                const int64_t base = ((int64_t)slot * p.kv_heads + kvh) * D;
#pragma unroll
                for (int cg = 0; cg < CH / 4; ++cg) {
                    const int c = cg * 4 + csub;
                    rc::cp_async16(rc::smem_u32(sK + tc::cm_offset(key, c, CH)), p.pool_k + base + c * 8, bytes);
                    rc::cp_async16(rc::smem_u32(sV + tc::cm_offset(key, c, CH)), p.pool_v + base + c * 8, bytes);
                }
            }
            rc::cp_async_commit();
            // hand over this warp's previous tile once its rows have landed
            if (prev >= 0) {
                rc::cp_async_wait<1>();
                tc::fence_proxy_async();
                mbar_arrive(&kv_full[prev % NS]);
            }
            prev = t;
            sl[0] = sl_next[0];
            sl[1] = sl_next[1];
        }
        rc::cp_async_wait<0>();
        tc::fence_proxy_async();
        if (ok && prev >= 0) mbar_arrive(&kv_full[prev % NS]);
        if (!ok) rc::flag_error(p.err, rc::kErrTimeout);
    } else if (lane == 0) {
        // ==================================================== MMA (warp 10)
        auto issue_s = [&](int t) {
            const uint32_t k0 = rc::smem_u32(sKV + (t % NS) * 2 * KV_BYTES);
            for (int q = 0; q < n_qt; ++q) {
                const uint32_t q0 = rc::smem_u32(sQ + q * TM * D * 2);
#pragma unroll
                for (int k = 0; k < D / 16; ++k)
                    tc::mma_bf16(tbase + q * 256 + (t & 1) * TN, tc::smem_desc(q0 + k * 256, 128, SB),
                                 tc::smem_desc(k0 + k * 256, 128, SB), idS, k > 0);
                tc::commit(&s_full[q * 2 + (t & 1)]);
            }
        };
        ok = tc::mbar_wait(q_full, 0, kWaitIter);
        if (ok && n_tiles > 0) {
            ok = tc::mbar_wait(&kv_full[0], 0, kWaitIter);
            tc::fence_after();
            if (ok) issue_s(0);
        }
        for (int t = 0; t < n_tiles && ok; ++t) {
            const int s = t % NS;
            if (t + 1 < n_tiles) {  // next tile's S products first: they run during this softmax
                ok = tc::mbar_wait(&kv_full[(t + 1) % NS], ((t + 1) / NS) & 1, kWaitIter);
                tc::fence_after();
                if (!ok) break;
                issue_s(t + 1);
            }
            const uint32_t v0 = rc::smem_u32(sKV + s * 2 * KV_BYTES + KV_BYTES);
            for (int q = 0; q < n_qt && ok; ++q) {
                ok = tc::mbar_wait(&p_full[q], t & 1, kWaitIter);
                tc::fence_after();
                if (!ok) break;
                const uint32_t p0 = rc::smem_u32(sP + q * TM * TN * 2);
#pragma unroll
                for (int j = 0; j < TN / 16; ++j)
                    tc::mma_bf16(tbase + q * 256 + 128, tc::smem_desc(p0 + j * 256, 128, (TN / 8) * 128),
                                 tc::smem_desc(v0 + j * 2 * SB, SB, 128), idPV, t > 0 || j > 0);
                tc::commit(&o_done[q]);
            }
            tc::commit(&kv_empty[s]);  // stage s is free once everything issued so far is done
        }
        if (!ok) rc::flag_error(p.err, rc::kErrTimeout);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 10) {
        tc::fence_after();
        tc::tmem_dealloc(tbase, 512);
    }
}

}  // namespace rc_tc2
