// Latent (MLA) decode on tcgen05 for 128 query heads: the 128 heads of one
// request are the M = 128 rows of the tensor-core products, so every latent
// row gathered serves all of them (the SGLang engineering article, section 1:
// with one KV head the decode kernel should serve many query heads per block;
// here a block serves all of them).
//
// CTA = (key chunk, value half, request).  Both value halves compute
// S = Q K^T over the full 576-wide key; each accumulates O for its 256 of the
// 512 value columns.  Q's first 384 columns are the A operand of S from
// tensor memory, its last 192 from shared memory: TMEM then holds two S
// buffers (columns 0 and 32, P over their first 16), Q (64..255) and O
// (256..511), and shared memory has room for four K/V stages next to the rest
// of Q.  Nine warps with fixed roles:
//   warps 0-3  softmax: one thread per head (TMEM lane); read S, write P (bf16)
//              back over it, rescale the head's O in TMEM when its max grows by
//              more than 2^8;
//   warps 4-7  producers, one per stage (tile t goes to stage t mod 4): gather
//              32 latent rows per tile by slot id with 16-byte cp.async
//              (no-swizzle core-matrix layout), each lane arriving on the
//              stage's barrier when its copies land, and asking L2 for the rows
//              of the warp's next tile one lap ahead;
//   warp 8     MMA issuer (one thread) and TMEM owner.
// Per 32-key tile: S = Q K^T (M 128, N 32, K 576 in 36 steps) into one of two
// S buffers; O += P V (M 128, N 256, K 32) with P read from TMEM and V the
// value half of the same shared-memory tile read as an MN-major operand.  The
// issuer never holds a ready P.V behind a tile that is still loading: it
// issues P(t).V as soon as the softmax hands P(t) over, and S(t+1) as soon as
// tile t+1 has landed, whichever comes first.  Every wait is bounded and
// flags RC_ERR_TIMEOUT when it gives up; a parity wait never has three
// possible phases (see the last-tile handling).
// The MMA thread and the producers issue back to back and share their
// sub-partitions with the other warps, so their instructions are kept few:
// the descriptors of a tile are built once and stepped along K by 32-bit
// adds, and a producer lane's 18 copies of a row carry their offsets as
// immediates (measured on the GB300: 1.78 -> 1.56 ms per full-size step).
#pragma once

#include "tc.cuh"

namespace rc_mla_tc {

constexpr int DK = 576, DV = 512, DVH = 256;
constexpr int M = 128;        // query heads per CTA (all)
constexpr int TN = 32;        // keys per tile
constexpr int NS = 4;         // K/V stages (one producer warp each)
constexpr int CK = DK / 8;    // 72 chunks of 16 bytes per latent row
constexpr int QT = 384;       // Q columns held in TMEM (24 K steps)
constexpr int CQ = (DK - QT) / 8;  // 24 chunks of Q per head in shared memory
constexpr int W_MMA = 4 + NS;      // warp index of the MMA issuer
constexpr int THREADS = 32 * (W_MMA + 1);
constexpr uint32_t COL_Q = 2 * TN, COL_O = 256;  // TMEM columns
constexpr int Q_BYTES = M * (DK - QT) * 2;
constexpr int TILE_BYTES = TN * DK * 2;
constexpr uint32_t SB = CK * 128;   // bytes between 8-row groups of a tile
constexpr uint32_t SBQ = CQ * 128;  // bytes between 8-head groups of Q
constexpr int kBars = 1 + 2 * NS + 2 + 2 + 1;
constexpr uint32_t kWaitIter = 1u << 24;
static_assert(COL_Q + QT / 2 <= COL_O, "Q and the S buffers overlap O in TMEM");

__host__ __device__ constexpr int smem_bytes() { return Q_BYTES + NS * TILE_BYTES + kBars * 8 + 16; }

struct Params {
    const __nv_bfloat16* q;      // [B][128][576]
    const __nv_bfloat16* pool;   // [n_slots][576]
    int64_t n_slots;
    float scale_log2;
    int32_t* err;
    const int32_t* table;
    const int32_t* start;
    const int32_t* len;
    int64_t table_len;
    int32_t chunk, n_chunks;     // keys per CTA, chunks per request
    float* part_o;               // [B][128][n_chunks][512] normalised partials
    float* part_lse;             // [B][128][n_chunks], log2 units, -inf: empty
    __nv_bfloat16* out;          // [B][128][512] (one chunk)
    float* lse;                  // [B][128] natural log, or NULL (one chunk)
};

template <bool FUSED>
__global__ void __launch_bounds__(THREADS, 1) mla_tc_kernel(const Params p) {
    constexpr uint32_t idS = tc::idesc_bf16(M, TN, false);
    constexpr uint32_t idPV = tc::idesc_bf16(M, DVH, true);
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* sQ = smem;                      // [128 heads][Q columns 384..575], no swizzle
    unsigned char* sKV = sQ + Q_BYTES;             // [NS][32 keys][576]
    uint64_t* bar = reinterpret_cast<uint64_t*>(sKV + NS * TILE_BYTES);
    uint64_t* q_full = bar + 0;                    // count 4 (softmax warps)
    uint64_t* kv_full = bar + 1;                   // [NS], count 32 (the stage's producer lanes, through cp.async)
    uint64_t* kv_empty = bar + 1 + NS;             // [NS], count 1 (MMA commit)
    uint64_t* s_full = bar + 1 + 2 * NS;           // [2], count 1
    uint64_t* p_full = s_full + 2;                 // [2], count 4
    uint64_t* o_done = p_full + 2;                 // count 1 per tile
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + kBars);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.y, chunk = blockIdx.x >> 1, vh = blockIdx.x & 1;
    const int64_t row0 = p.start[b];
    int L = p.len[b];
    if (row0 < 0 || L < 0 || row0 + L > p.table_len) {
        if (tid == 0 && chunk == 0 && vh == 0) rc::flag_error(p.err, rc::kErrBadSlot);
        L = 0;
    }
    if (FUSED && L > p.chunk) {
        if (tid == 0 && vh == 0) rc::flag_error(p.err, rc::kErrBadSlot);
        L = p.chunk;
    }
    const int k0 = chunk * p.chunk;
    const int count = min(L - k0, p.chunk);
    if (count <= 0) {  // nothing here: an empty partial (or, fused, an empty row)
        if (tid < M) {
            const int64_t bh = (int64_t)b * M + tid;
            if constexpr (FUSED) {
                for (int c = 0; c < DVH; c += 8)
                    *reinterpret_cast<uint4*>(p.out + bh * DV + vh * DVH + c) = make_uint4(0, 0, 0, 0);
                if (p.lse && vh == 0) p.lse[bh] = -INFINITY;
            } else if (vh == 0) {
                p.part_lse[bh * p.n_chunks + chunk] = -INFINITY;
            }
        }
        return;
    }
    // one decision for the whole CTA: the word can change between two
    // threads' reads, and a CTA split here would stall at its first barrier
    if (__syncthreads_or(p.err && (*reinterpret_cast<volatile int32_t*>(p.err) & rc::kErrTimeout))) return;
    const int32_t* keys = p.table + row0 + k0;
    const int n_tiles = (count + TN - 1) / TN;

    // producer: slot ids of the first tile, before the set-up
    int sl = -1;
    if (warp >= 4 && warp < W_MMA && (warp - 4) * TN + lane < count) sl = __ldg(keys + (warp - 4) * TN + lane);
    const __nv_bfloat16* qb = p.q + (int64_t)b * M * DK;
    if (warp < 4) {
        // Q columns 384..575 of all 128 heads: 8 consecutive lanes write 8
        // rows of one 16-byte column, 128 contiguous bytes of the core-matrix
        // layout
        for (int gi = tid; gi < M * CQ; gi += 128) {
            const int j = gi & 7, rest = gi >> 3;
            const int c = rest % CQ, rg = rest / CQ;
            const int r = rg * 8 + j;
            rc::cp_async16(rc::smem_u32(sQ + tc::cm_offset(r, c, CQ)), qb + (int64_t)r * DK + QT + c * 8, 16u);
        }
        rc::cp_async_commit();
    }
    if (tid == 0) {
        tc::mbar_init(q_full, 4);
        for (int s = 0; s < NS; ++s) {
            tc::mbar_init(&kv_full[s], 32);
            tc::mbar_init(&kv_empty[s], 1);
        }
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&s_full[i], 1);
            tc::mbar_init(&p_full[i], 4);
        }
        tc::mbar_init(o_done, 1);
        tc::fence_mbar_init();
    }
    if (warp == W_MMA) {
        tc::tmem_alloc(tslot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tbase = *tslot;
    bool ok = true;

    if (warp < 4) {
        // ================================================ softmax (one head per thread)
        const uint32_t tl = tbase + ((uint32_t)(warp * 32) << 16);
        const uint32_t tO = tl + COL_O;
        {
            // Q columns 0..383 of this thread's head into its TMEM lane, two
            // bf16 per column (the even column in the low half), 64 per store
            const uint4* qrow = reinterpret_cast<const uint4*>(qb + (int64_t)tid * DK);
#pragma unroll 1
            for (int g = 0; g < QT / 64; ++g) {
                uint32_t r[32];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 v = __ldg(qrow + g * 8 + i);
                    r[4 * i] = v.x;
                    r[4 * i + 1] = v.y;
                    r[4 * i + 2] = v.z;
                    r[4 * i + 3] = v.w;
                }
                tc::tmem_st32_issue(tl + COL_Q + g * 32, r);
                tc::tmem_st_wait();
            }
        }
        rc::cp_async_wait<0>();
        tc::fence_proxy_async();
        tc::fence_before();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(q_full);
        const float sc = p.scale_log2;
        float m_used = -INFINITY, l_run = 0.f;
        for (int t = 0; t < n_tiles && ok; ++t) {
            ok = __all_sync(0xffffffffu, tc::mbar_wait(&s_full[t & 1], (t >> 1) & 1, kWaitIter));
            tc::fence_after();
            const uint32_t tS = tl + (t & 1) * TN;
            uint32_t sr[32];
            tc::tmem_ld32_issue(tS, sr);
            tc::tmem_ld_wait(sr);
            float s[TN];
#pragma unroll
            for (int j = 0; j < TN; ++j) s[j] = __uint_as_float(sr[j]);
            const int kb = t * TN;
            if (kb + TN > count) {
#pragma unroll
                for (int j = 0; j < TN; ++j)
                    if (kb + j >= count) s[j] = -INFINITY;
            }
            float m4[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                m4[i] = tc::max3(s[i], s[4 + i], s[8 + i]);
                m4[i] = tc::max3(m4[i], s[12 + i], s[16 + i]);
                m4[i] = tc::max3(m4[i], s[20 + i], s[24 + i]);
                m4[i] = fmaxf(m4[i], s[28 + i]);
            }
            const float mt = tc::max3(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sc;
            const bool grow = mt > m_used + 8.f;
            const bool rescale_o = grow && m_used != -INFINITY;
            if (__any_sync(0xffffffffu, rescale_o)) {
                // O must be stable: P(t-1).V is done (S(t) guarantees P(t-2).V)
                ok = __all_sync(0xffffffffu, tc::mbar_wait(o_done, (t - 1) & 1, kWaitIter)) && ok;
                tc::fence_after();
                const float a = rescale_o ? tc::ex2(m_used - mt) : 1.f;
#pragma unroll 1
                for (int c = 0; c < DVH / 32; ++c) {
                    uint32_t v[32];
                    tc::tmem_ld32_issue(tO + c * 32, v);
                    tc::tmem_ld_wait(v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = __float_as_uint(__uint_as_float(v[j]) * a);
                    tc::tmem_st32_issue(tO + c * 32, v);
                }
                tc::tmem_st_wait();
            }
            if (grow) {
                l_run *= tc::ex2(m_used - mt);
                m_used = mt;
            }
            const float nmu = m_used == -INFINITY ? 0.f : -m_used;
            uint32_t pk[16];
            float2 ls[2] = {{0.f, 0.f}, {0.f, 0.f}};
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float2 x = tc::ffma2(make_float2(s[2 * i], s[2 * i + 1]), sc, nmu);
                const float2 e = make_float2(tc::ex2(x.x), tc::ex2(x.y));
                ls[i & 1] = tc::fadd2(ls[i & 1], e);
                pk[i] = rc::pack_bf16(e.x, e.y);
            }
            tc::tmem_st16_issue(tS, pk);
            const float2 l2 = tc::fadd2(ls[0], ls[1]);
            l_run += l2.x + l2.y;
            tc::tmem_st_wait();
            if (t == n_tiles - 1 && t > 0) {  // last tile: P(n-2).V done before P(n-1) goes
                ok = __all_sync(0xffffffffu, tc::mbar_wait(o_done, (t - 1) & 1, kWaitIter)) && ok;
                tc::fence_after();
            }
            tc::fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&p_full[t & 1]);
        }
        if (ok) ok = __all_sync(0xffffffffu, tc::mbar_wait(o_done, (n_tiles - 1) & 1, kWaitIter));
        tc::fence_after();
        if (!ok) rc::flag_error(p.err, rc::kErrTimeout);
        // ---- epilogue: this CTA's 256 value columns of every head.  Each
        // warp's 32x32 fp32 blocks go through its 4 KB of the (now free) Q
        // region, so stores write whole row segments.
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        const float lse2 = l_run > 0.f ? m_used + log2f(l_run) : -INFINITY;
        float* stg = reinterpret_cast<float*>(sQ + warp * 4096);
        const int k8 = lane & 7;
#pragma unroll 1
        for (int c = 0; c < DVH / 32; ++c) {
            uint32_t vb[32];
            tc::tmem_ld32_issue(tO + c * 32, vb);
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
                const int64_t bh = (int64_t)b * M + warp * 32 + rr;
                const int col = vh * DVH + c * 32 + k8 * 4;
                if (!ok) continue;
                if constexpr (FUSED) {
                    uint2 w;
                    w.x = rc::pack_bf16(f.x, f.y);
                    w.y = rc::pack_bf16(f.z, f.w);
                    *reinterpret_cast<uint2*>(p.out + bh * DV + col) = w;
                } else {
                    *reinterpret_cast<float4*>(p.part_o + (bh * p.n_chunks + chunk) * DV + col) = f;
                }
            }
            __syncwarp();
        }
        if (ok && vh == 0) {
            const int64_t bh = (int64_t)b * M + tid;
            if constexpr (FUSED) {
                if (p.lse) p.lse[bh] = lse2 * rc::kLn2;
            } else {
                p.part_lse[bh * p.n_chunks + chunk] = lse2;
            }
        }
    } else if (warp < W_MMA) {
        // ================================================ producers (stage = warp - 4)
        // lane -> (key within an 8-key group, 16-byte column within a group
        // of 4): 8 lanes write 128 contiguous bytes of the core-matrix layout
        const int klo = lane & 7, csub = lane >> 3;
        const int s = warp - 4;
        for (int t = s; t < n_tiles && ok; t += NS) {
            int sl_next = -1;
            {
                const int key = (t + NS) * TN + lane;
                if (t + NS < n_tiles && key < count) sl_next = __ldg(keys + key);
            }
            if (t >= NS) ok = __all_sync(0xffffffffu, tc::mbar_wait(&kv_empty[s], ((t / NS) + 1) & 1, kWaitIter));
            if (!ok) break;
            unsigned char* sT = sKV + s * TILE_BYTES;
#pragma unroll
            for (int kg = 0; kg < TN / 8; ++kg) {
                const int key = kg * 8 + klo;
                int slot = __shfl_sync(0xffffffffu, sl, key);
                uint32_t bytes = 16;
                if (t * TN + key >= count) { slot = 0; bytes = 0; }
                else if (slot < 0 || (int64_t)slot >= p.n_slots) {
                    rc::flag_error(p.err, rc::kErrBadSlot);
                    slot = 0;
                    bytes = 0;
                }
                // chunks c = 4 cg + csub: 512 bytes apart in the stage, 64 in the row
                const __nv_bfloat16* src = p.pool + (int64_t)slot * DK + csub * 8;
                rc::cp_async16_run<512, 64>(rc::smem_u32(sT + tc::cm_offset(key, csub, CK)), src, bytes,
                                            std::make_integer_sequence<int, CK / 4>{});
            }
            tc::cp_async_mbar_arrive(&kv_full[s]);
            // the rows of this warp's next tile (NS tiles on) start for L2 now
            if (sl_next >= 0 && (int64_t)sl_next < p.n_slots)
                rc::prefetch_l2(p.pool + (int64_t)sl_next * DK, (uint32_t)(DK * 2));
            sl = sl_next;
        }
        rc::cp_async_wait<0>();
        if (!ok) rc::flag_error(p.err, rc::kErrTimeout);
    } else if (lane == 0) {
        // ================================================ MMA (one thread)
        const uint32_t q0 = rc::smem_u32(sQ);
        const tc::Desc qd = tc::desc_halves(q0, 128, SBQ);
        auto issue_s = [&](int t) {
            const tc::Desc kd = tc::desc_halves(rc::smem_u32(sKV + (t % NS) * TILE_BYTES), 128, SB);
            const uint32_t d = tbase + (t & 1) * TN;
            // Q columns 0..QT-1 from TMEM (8 columns per K step of 16), K
            // steps 256 bytes apart in both operands
#pragma unroll
            for (int k = 0; k < QT / 16; ++k)
                tc::mma_bf16_ts_h(d, tbase + COL_Q + k * 8, kd.lo + k * 16, kd.hi, idS, k > 0);
            // the rest of Q from shared memory
#pragma unroll
            for (int k = 0; k < (DK - QT) / 16; ++k)
                tc::mma_bf16_h(d, qd.lo + k * 16, qd.hi, kd.lo + (QT / 16 + k) * 16, kd.hi, idS, 1u);
            tc::commit(&s_full[t & 1]);
        };
        ok = tc::mbar_wait(q_full, 0, kWaitIter);
        tc::fence_after();
        // t: next P.V to issue; ns: S products issued.  S(ns) may go once
        // P(ns-2).V is issued (it overwrites that S buffer), i.e. ns <= t + 1.
        int ns = 0;
        uint32_t idle = 0;
        uint64_t t0 = 0;
        for (int t = 0; t < n_tiles && ok;) {
            bool moved = false;
            if (ns > t && tc::mbar_test(&p_full[t & 1], (t >> 1) & 1)) {
                tc::fence_after();
                // value half vh of the tile: columns [256 vh, 256 vh + 256) = chunks [32 vh, 32 vh + 32)
                const int s = t % NS;
                const tc::Desc vd =
                    tc::desc_halves(rc::smem_u32(sKV + s * TILE_BYTES) + vh * (DVH / 8) * 128, SB, 128);
#pragma unroll
                for (int j = 0; j < TN / 16; ++j)
                    tc::mma_bf16_ts_h(tbase + COL_O, tbase + (t & 1) * TN + j * 8, vd.lo + j * (2 * SB / 16), vd.hi,
                                      idPV, (t > 0 || j > 0) ? 1u : 0u);
                tc::commit(o_done);
                tc::commit(&kv_empty[s]);
                ++t;
                moved = true;
            }
            if (ns < n_tiles && ns <= t + 1 && tc::mbar_test(&kv_full[ns % NS], (ns / NS) & 1)) {
                tc::fence_after();
                tc::fence_proxy_async();  // the rows arrived through the generic proxy
                issue_s(ns);
                ++ns;
                moved = true;
            }
            if (moved) {
                idle = 0;
                t0 = 0;
                continue;
            }
            // nothing ready: probe again at once (a sleep here costs more than
            // the softmax hand-off it waits for)
            if ((++idle & 1023) == 0) {
                uint64_t now;
                asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(now));
                if (t0 == 0) t0 = now;
                else if (now - t0 > tc::kWaitNs || idle >= kWaitIter) ok = false;
            }
        }
        if (!ok) rc::flag_error(p.err, rc::kErrTimeout);
    }
    tc::fence_before();
    __syncthreads();
    if (warp == W_MMA) {
        tc::fence_after();
        tc::tmem_dealloc(tbase, 512);
    }
}

// Grid (2 x chunks, batch): x = chunk * 2 + value half.
template <bool FUSED>
cudaError_t launch(const Params& t, int n_chunks, int batch, cudaStream_t st) {
    constexpr int smem = smem_bytes();
    cudaError_t e = rc_host::ensure_smem<mla_tc_kernel<FUSED>>(smem);
    if (e != cudaSuccess) return e;
    mla_tc_kernel<FUSED><<<dim3(2 * n_chunks, batch), THREADS, smem, st>>>(t);
    return cudaGetLastError();
}

}  // namespace rc_mla_tc
