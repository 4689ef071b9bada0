// Many query rows over one gathered key list on the fifth-generation tensor
// cores (tcgen05, accumulators in TMEM): the kernel body of attn_extend (new
// tokens over their cached prefix, causal among themselves) and of the
// cascade step of attn_decode (a shared segment read once for every request
// below it).
//
// CTA = 128 query rows of one KV head = (128/G tokens or requests) x (the G
// query heads of that KV head), the M of both products.  Per 64-key tile:
//   S = Q K^T   (M=128, N=64, K=head dim)  -> TMEM columns [0, 64) or [64, 128)
//   O += P V    (M=128, N=head dim, K=64)  -> TMEM columns [128, 128 + D)
// S is double-buffered: S of the next tile is issued before this tile's
// softmax, so the tensor core works on it (and on the previous P.V) meanwhile.
// One thread issues the MMAs and commits each product to an mbarrier; every
// thread owns one TMEM lane (one query row) for the online softmax: it reads
// its S row, writes its P row (bf16) to shared memory in the operand layout,
// and rescales its O row in TMEM only when its running max has grown by more
// than 2^8 since the last rescale (p then stays below 2^8, exact in fp32).
// K/V rows are gathered by slot id with 16-byte cp.async straight into the
// operand layout (tc.cuh); slot ids ride the same pipeline ahead of the rows.
// About 113 KB of shared memory and 256 TMEM columns: two CTAs per SM, whose
// softmax phases overlap each other's MMAs.
#pragma once

#include "mq_attn.cuh"
#include "tc.cuh"

namespace rc_tc {

constexpr int TM = 128;   // query rows per CTA
constexpr int TN = 64;    // keys per tile
constexpr int RING = 3;   // tiles of slot ids
constexpr uint32_t kWaitIter = 1u << 24;

template <int D>
__host__ __device__ constexpr int smem_bytes() {
    return TM * D * 2 + 2 * TN * D * 2 + 2 * TN * D * 2 + TM * TN * 2 + RING * TN * 4 + 64 + 16;
}
template <int D>
__host__ __device__ constexpr uint32_t tmem_cols() {  // two S buffers [0, 128) + O [128, 128 + D)
    return 256u;
}

template <int D, int G, rc::MQMode MODE>
__global__ void __launch_bounds__(128, 2) attn_tc_kernel(const rc::MQParams p) {
    constexpr int CH = D / 8;
    constexpr int TPC = TM / G;
    constexpr int KV_BYTES = TN * D * 2;
    constexpr int PER = TN * CH / 128;     // 16-byte chunks per thread per K (or V) tile
    constexpr uint32_t kO = 128u;
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* sQ = smem;
    unsigned char* sK = sQ + TM * D * 2;
    unsigned char* sV = sK + 2 * KV_BYTES;
    unsigned char* sP = sV + 2 * KV_BYTES;
    int32_t* sSlot = reinterpret_cast<int32_t*>(sP + TM * TN * 2);
    uint64_t* mbar = reinterpret_cast<uint64_t*>(sSlot + RING * TN);   // [0], [1]: S buffers; [2]: P.V
    uint32_t* tslot = reinterpret_cast<uint32_t*>(mbar + 3);
    int* sAbort = reinterpret_cast<int*>(tslot + 1);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int kvh = blockIdx.y, z = blockIdx.z, blk = blockIdx.x;
    const int tok0 = blk * TPC;

    // ---- this CTA's rows and keys
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
            const int tk = tok0 + tid / G;
            if (tk < n_rows_tok)
                p.part_lse[((int64_t)(qo0 + tk) * p.q_heads + kvh * G + (tid % G)) * p.seg_chunks + chunk] =
                    -INFINITY;
            return;
        }
    }
    const int n_tiles = (key_count + TN - 1) / TN;

    // ---- loaders (thread mapping: the 8 rows of a core matrix are 8
    // consecutive threads, so each warp writes whole 128-byte core matrices)
    auto copy_slots = [&](int kt) {
        if (tid < TN) {
            const int key = kt * TN + tid;
            const bool ok = kt < n_tiles && key < key_count;
            rc::cp_async4(rc::smem_u32(sSlot + (kt % RING) * TN + tid), ok ? keys + key : keys, ok ? 4u : 0u);
        }
    };
    auto gather = [&](int kt, unsigned char* dst, const __nv_bfloat16* pool) {
        if (kt >= n_tiles) return;
        const int32_t* ring = sSlot + (kt % RING) * TN;
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int gi = i * 128 + tid;
            const int r = (gi & 7) + 8 * (gi / (8 * CH));
            const int c = (gi >> 3) % CH;
            int slot = ring[r];
            uint32_t bytes = 16;
            if (kt * TN + r >= key_count) { slot = 0; bytes = 0; }
            else if (slot < 0 || (int64_t)slot >= p.n_slots) {
                rc::flag_error(p.err, rc::kErrBadSlot);
                slot = 0;
                bytes = 0;
            }
            rc::cp_async16(rc::smem_u32(dst + tc::cm_offset(r, c, CH)),
                           pool + ((int64_t)slot * p.kv_heads + kvh) * D + c * 8, bytes);
        }
    };

    // ---- prologue: slot ids of tiles 0..2; then groups {Q, K0}, {K1}, {V0}.
    // Each iteration kt then commits {K(kt+2), ids(kt+3)} and {V(kt+1)}, so at
    // the top of iteration kt K(kt+1) is in the second-newest group (wait<1>)
    // and before its P.V, V(kt) is third-newest (wait<2>).
    for (int t = 0; t < 3; ++t) copy_slots(t);
    rc::cp_async_commit();
    rc::cp_async_wait<0>();
    __syncthreads();
    for (int gi = tid; gi < TM * CH; gi += 128) {
        const int r = (gi & 7) + 8 * (gi / (8 * CH));
        const int c = (gi >> 3) % CH;
        const int tk = tok0 + r / G;
        const int h = kvh * G + (r % G);
        int64_t qrow = 0;
        if (tk < n_rows_tok) {
            if constexpr (MODE == rc::MQMode::kExtend) qrow = (int64_t)(qo0 + tk) * p.q_heads + h;
            else qrow = (int64_t)p.seg_rows[qo0 + tk] * p.q_heads + h;
        }
        rc::cp_async16(rc::smem_u32(sQ + tc::cm_offset(r, c, CH)), p.q + qrow * D + c * 8,
                       tk < n_rows_tok ? 16u : 0u);
    }
    gather(0, sK, p.pool_k);
    rc::cp_async_commit();
    gather(1, sK + KV_BYTES, p.pool_k);
    rc::cp_async_commit();
    gather(0, sV, p.pool_v);
    rc::cp_async_commit();

    if (warp == 0) {
        tc::tmem_alloc(tslot, tmem_cols<D>());
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(&mbar[0], 1);
        tc::mbar_init(&mbar[1], 1);
        tc::mbar_init(&mbar[2], 1);
        tc::fence_mbar_init();
        *sAbort = 0;
    }
    rc::cp_async_wait<2>();   // Q and K0
    tc::fence_proxy_async();
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tbase = *tslot;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t tO = tbase + kO + lane_off;

    const int r_tok = tok0 + tid / G;
    const bool row_valid = r_tok < n_rows_tok;
    int lim;
    if constexpr (MODE == rc::MQMode::kExtend) lim = row_valid ? prefix + r_tok + 1 : 0;
    else lim = row_valid ? key_count : 0;
    float m_used = -INFINITY, l_run = 0.f;
    constexpr uint32_t idS = tc::idesc_bf16(TM, TN, false);
    constexpr uint32_t idPV = tc::idesc_bf16(TM, D, true);
    constexpr uint32_t SB = CH * 128;   // bytes between 8-row groups of a Q/K/V tile

    // S(t) = Q K(t)^T into TMEM buffer t&1 (columns 64*(t&1)), committed to mbar[t&1]
    auto issue_s = [&](int t) {
        tc::fence_after();
        const uint32_t q0 = rc::smem_u32(sQ), k0 = rc::smem_u32(sK + (t & 1) * KV_BYTES);
#pragma unroll
        for (int k = 0; k < D / 16; ++k)
            tc::mma_bf16(tbase + (t & 1) * TN, tc::smem_desc(q0 + k * 256, 128, SB),
                         tc::smem_desc(k0 + k * 256, 128, SB), idS, k > 0);
        tc::commit(&mbar[t & 1]);
    };
    if (tid == 0) issue_s(0);

    int kt = 0;
    for (; kt < n_tiles; ++kt) {
        const int st = kt & 1;
        // K(kt+1) has landed (second-newest group): start S(kt+1) now so the
        // tensor core works while this tile's softmax runs
        rc::cp_async_wait<1>();
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        if (*sAbort) break;
        if (tid == 0 && kt + 1 < n_tiles) issue_s(kt + 1);
        bool ok = tc::mbar_wait(&mbar[st], (kt >> 1) & 1, kWaitIter);
        tc::fence_after();
        float s[TN];
        const uint32_t tS = tbase + st * TN + lane_off;
        tc::tmem_ld32(tS, *reinterpret_cast<float(*)[32]>(&s[0]));
        tc::tmem_ld32(tS + 32, *reinterpret_cast<float(*)[32]>(&s[32]));
        const int kb = kt * TN;
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < TN; ++j) {
            s[j] = kb + j < lim ? s[j] * p.scale_log2 : -INFINITY;
            mt = fmaxf(mt, s[j]);
        }
        // the previous P.V must be done before O, P and V(kt-1) are touched
        if (kt > 0) {
            ok = tc::mbar_wait(&mbar[2], (kt - 1) & 1, kWaitIter) && ok;
            tc::fence_after();
        }
        if (!ok) {
            rc::flag_error(p.err, rc::kErrTimeout);
            *sAbort = 1;
        }
        // K(kt)'s stage is free (S(kt) done), V(kt-1)'s too (P.V(kt-1) done): refill
        gather(kt + 2, sK + st * KV_BYTES, p.pool_k);
        copy_slots(kt + 3);
        rc::cp_async_commit();
        gather(kt + 1, sV + (st ^ 1) * KV_BYTES, p.pool_v);
        rc::cp_async_commit();
        if (mt > m_used + 8.f) {
            if (kt > 0 && m_used != -INFINITY) {  // bring O and l to the new max
                const float a = rc::fast_exp2(m_used - mt);
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    float v[32];
                    tc::tmem_ld32(tO + c * 32, v);
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] *= a;
                    tc::tmem_st32(tO + c * 32, v);
                }
                l_run *= a;
            }
            m_used = mt;
        }
        // P row (bf16) in the A-operand layout: 8 chunks of 8 keys
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
            *reinterpret_cast<uint4*>(sP + tc::cm_offset(tid, c, TN / 8)) = w;
        }
        // V(kt) must have landed: third-newest group
        rc::cp_async_wait<2>();
        tc::fence_proxy_async();
        tc::fence_before();
        __syncthreads();
        if (tid == 0) {  // O += P V
            tc::fence_after();
            const uint32_t p0 = rc::smem_u32(sP), v0 = rc::smem_u32(sV + st * KV_BYTES);
#pragma unroll
            for (int j = 0; j < TN / 16; ++j)
                tc::mma_bf16(tbase + kO, tc::smem_desc(p0 + j * 256, 128, (TN / 8) * 128),
                             tc::smem_desc(v0 + j * 2 * SB, SB, 128), idPV, kt > 0 || j > 0);
            tc::commit(&mbar[2]);
        }
    }
    const int done_tiles = kt;
    if (done_tiles > 0 && !tc::mbar_wait(&mbar[2], (done_tiles - 1) & 1, kWaitIter))
        rc::flag_error(p.err, rc::kErrTimeout);
    tc::fence_after();
    rc::cp_async_wait<0>();

    // ---- epilogue: normalised O row (and its log-sum-exp)
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    const float lse2 = l_run > 0.f ? m_used + log2f(l_run) : -INFINITY;
    const bool write = row_valid && done_tiles == n_tiles;
    const int h = kvh * G + (tid % G);
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
        float v[32];
        tc::tmem_ld32(tO + c * 32, v);
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
            float* dst = p.part_o + (((int64_t)(qo0 + r_tok) * p.q_heads + h) * p.seg_chunks + chunk) * D + c * 32;
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
    tc::fence_before();
    __syncthreads();
    if (warp == 0) tc::tmem_dealloc(tbase, tmem_cols<D>());
}

}  // namespace rc_tc
