// Many query rows over one gathered key list: the shared kernel body of
// attn_extend (new tokens over their cached prefix, causal among themselves)
// and of the cascade step of attn_decode (a shared prefix segment read once
// for every request that branches below it).
//
// A CTA owns 64 query rows of one KV head: (token or request) x (the G query
// heads of that KV head), so each K/V row fetched from HBM serves G heads and
// up to 64/G tokens at once.  K/V rows are gathered by slot id with 16-byte
// cp.async into an XOR-swizzled shared-memory ring of 64-key tiles; the two
// products run on the tensor cores (mma.sync m16n8k16 bf16, fp32
// accumulate); softmax is online (running max and sum per row, rescaling the
// output accumulators), exactly as in flash attention.
#pragma once

#include "common.cuh"

namespace rc {

enum class MQMode { kExtend, kCascade };

struct MQParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* pool_k;
    const __nv_bfloat16* pool_v;
    int64_t n_slots;
    int32_t kv_heads, q_heads;
    float scale_log2;  // sm_scale * log2(e)
    int32_t* err;
    // extend: rows are new tokens of request blockIdx.z
    const int32_t* qo_indptr;
    const int32_t* table;
    const int32_t* start;
    const int32_t* len;
    int64_t table_len;
    __nv_bfloat16* out;
    float* lse;
    // cascade: rows are the requests sharing segment blockIdx.z
    const int32_t* seg_slots;
    const int32_t* seg_indptr;
    const int32_t* seg_row_indptr;
    const int32_t* seg_rows;
    float* part_o;    // [total_seg_rows][q_heads][seg_chunks][D]
    float* part_lse;  // [total_seg_rows][q_heads][seg_chunks], log2 units (-inf: empty chunk)
    int32_t seg_chunk;   // keys per cascade CTA
    int32_t seg_chunks;  // chunks per segment (grid z = segment * seg_chunks + chunk)
};

constexpr int kMQRows = 64;
constexpr int kMQKeys = 64;
constexpr int kMQStages = 3;

constexpr int kMQSlotRing = 4;  // tiles of slot ids: written 4 ahead into the entry of the tile issued 2 iterations ago

template <int D>
__host__ __device__ constexpr int mq_smem_bytes() {
    return kMQRows * D * 2 + kMQStages * 2 * kMQKeys * D * 2 + kMQSlotRing * kMQKeys * 4;
}

template <int D, int G, MQMode MODE>
__global__ void __launch_bounds__(128, 2) mq_attn_kernel(const MQParams p) {
    constexpr int CH = D / 8;          // 16-byte chunks per row
    constexpr int TPC = kMQRows / G;   // tokens (or requests) per CTA
    constexpr int KS = D / 16;         // k-steps of the QK product
    constexpr int NT = D / 8;          // n-tiles of the output
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* sQ = smem;
    unsigned char* sKV = smem + kMQRows * D * 2;
    constexpr int TILE_BYTES = kMQKeys * D * 2;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g_lane = lane >> 2, t_lane = lane & 3;
    const int kvh = blockIdx.y;
    const int z = blockIdx.z;
    const int blk = blockIdx.x;

    // ---- this CTA's rows and key list
    int n_rows_tok;           // valid tokens/requests of the whole job
    int key_count;            // keys the CTA must visit
    const int32_t* keys;      // slot ids, position order
    int tok0 = blk * TPC;     // first token/request of this CTA
    int prefix = 0;           // extend: cached prefix length (position of new token 0)
    int qo0 = 0;
    if constexpr (MODE == MQMode::kExtend) {
        qo0 = p.qo_indptr[z];
        n_rows_tok = p.qo_indptr[z + 1] - qo0;
        const int L = p.len[z];
        prefix = L - n_rows_tok;
        const int64_t row0 = p.start[z];
        if (tok0 >= n_rows_tok) return;
        if (row0 < 0 || prefix < 0 || row0 + L > p.table_len) {  // row outside the table: read nothing
            if (tid == 0) flag_error(p.err, kErrBadSlot);
            return;
        }
        keys = p.table + row0;
        const int last = min(n_rows_tok, tok0 + TPC) - 1;
        key_count = prefix + last + 1;
    } else {
        const int seg = z / p.seg_chunks;
        const int chunk = z % p.seg_chunks;
        const int r0 = p.seg_row_indptr[seg];
        n_rows_tok = p.seg_row_indptr[seg + 1] - r0;
        qo0 = r0;
        const int k0 = chunk * p.seg_chunk;
        keys = p.seg_slots + p.seg_indptr[seg] + k0;
        key_count = min(p.seg_indptr[seg + 1] - p.seg_indptr[seg] - k0, p.seg_chunk);
        if (tok0 >= n_rows_tok) return;
        if (key_count <= 0) {  // segment shorter than this chunk: an empty partial
            for (int r = tid; r < kMQRows; r += 128) {
                const int tk = tok0 + r / G;
                if (tk < n_rows_tok)
                    p.part_lse[((int64_t)(qo0 + tk) * p.q_heads + kvh * G + (r % G)) * p.seg_chunks + chunk] =
                        -INFINITY;
            }
            return;
        }
    }

    int32_t* sSlot = reinterpret_cast<int32_t*>(sKV + kMQStages * 2 * TILE_BYTES);  // [ring][64]
    const int n_tiles = (key_count + kMQKeys - 1) / kMQKeys;

    // Slot ids travel through the cp.async pipeline: the group committed at
    // iteration kt holds K/V of tile kt+2 and the slot ids of tile kt+4, so a
    // gather never waits on the load of its own ids.
    auto copy_slots = [&](int kt) {
        if (tid < kMQKeys) {
            const int key = kt * kMQKeys + tid;
            const bool ok = kt < n_tiles && key < key_count;
            cp_async4(smem_u32(sSlot + (kt % kMQSlotRing) * kMQKeys + tid), ok ? keys + key : keys, ok ? 4u : 0u);
        }
    };
    auto load_tile = [&](int kt) {
        if (kt >= n_tiles) return;
        unsigned char* sK = sKV + (kt % kMQStages) * 2 * TILE_BYTES;
        unsigned char* sV = sK + TILE_BYTES;
        const int32_t* ring = sSlot + (kt % kMQSlotRing) * kMQKeys;
        constexpr int PER = kMQKeys * CH / 128;  // chunks per thread per matrix
#pragma unroll
        for (int i = 0; i < PER; ++i) {
            const int lin = i * 128 + tid;
            const int r = lin / CH, c = lin % CH;
            int slot = ring[r];
            uint32_t bytes = 16;
            if (kt * kMQKeys + r >= key_count) { slot = 0; bytes = 0; }
            else if (slot < 0 || (int64_t)slot >= p.n_slots) {
                flag_error(p.err, kErrBadSlot);
                slot = 0;
                bytes = 0;
            }
            const int64_t roff = ((int64_t)slot * p.kv_heads + kvh) * D + c * 8;
            cp_async16(smem_u32(sK + swz<CH>(r, c)), p.pool_k + roff, bytes);
            cp_async16(smem_u32(sV + swz<CH>(r, c)), p.pool_v + roff, bytes);
        }
    };

    // prologue: slot ids of tiles 0..3; then Q rows (zero past the end) + tile 0; tile 1
#pragma unroll
    for (int t = 0; t < 4; ++t) copy_slots(t);
    cp_async_commit();
    cp_async_wait<0>();
    __syncthreads();
    for (int i = tid; i < kMQRows * CH; i += 128) {
        const int r = i / CH, c = i % CH;
        const int tk = tok0 + r / G;
        const int h = kvh * G + (r % G);
        int64_t qrow = 0;
        if (tk < n_rows_tok) {
            if constexpr (MODE == MQMode::kExtend) qrow = (int64_t)(qo0 + tk) * p.q_heads + h;
            else qrow = (int64_t)p.seg_rows[qo0 + tk] * p.q_heads + h;
        }
        cp_async16(smem_u32(sQ + swz<CH>(r, c)), p.q + qrow * D + c * 8, tk < n_rows_tok ? 16u : 0u);
    }
    load_tile(0);
    cp_async_commit();
    load_tile(1);
    cp_async_commit();
    cp_async_wait<1>();
    __syncthreads();

    // ---- Q fragments of this warp's 16 rows
    uint32_t qa[KS][4];
    {
        const int r = warp * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
            ldmatrix_x4(smem_u32(sQ + swz<CH>(r, ks * 2 + (lane >> 4))), qa[ks][0], qa[ks][1], qa[ks][2],
                        qa[ks][3]);
    }

    // key limit of the two rows this thread holds (g and g+8 of the warp)
    int lim[2];
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int r = warp * 16 + g_lane + hr * 8;
        const int tk = tok0 + r / G;
        if constexpr (MODE == MQMode::kExtend) lim[hr] = tk < n_rows_tok ? prefix + tk + 1 : 0;
        else lim[hr] = tk < n_rows_tok ? key_count : 0;
    }

    float o[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    for (int kt = 0; kt < n_tiles; ++kt) {
        if (kt > 0) {
            cp_async_wait<1>();
            __syncthreads();
        }
        load_tile(kt + 2);
        copy_slots(kt + 4);
        cp_async_commit();
        const unsigned char* sK = sKV + (kt % kMQStages) * 2 * TILE_BYTES;
        const unsigned char* sV = sK + TILE_BYTES;

        float s[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) s[i][0] = s[i][1] = s[i][2] = s[i][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
            for (int n2 = 0; n2 < 4; ++n2) {
                uint32_t b0, b1, b2, b3;
                const int key = n2 * 16 + (lane & 7) + (lane >> 4) * 8;
                ldmatrix_x4(smem_u32(sK + swz<CH>(key, ks * 2 + ((lane >> 3) & 1))), b0, b1, b2, b3);
                mma_bf16_16816(s[2 * n2], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
                mma_bf16_16816(s[2 * n2 + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
            }
        }
        // mask, scale, running max
        const int kbase = kt * kMQKeys;
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int hr = e >> 1;
                const int key = kbase + nt * 8 + 2 * t_lane + (e & 1);
                const float v = key < lim[hr] ? s[nt][e] * p.scale_log2 : -INFINITY;
                s[nt][e] = v;
                mx[hr] = fmaxf(mx[hr], v);
            }
        }
        float alpha[2];
#pragma unroll
        for (int hr = 0; hr < 2; ++hr) {
            mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 1));
            mx[hr] = fmaxf(mx[hr], __shfl_xor_sync(0xffffffffu, mx[hr], 2));
            const float m_new = fmaxf(m_run[hr], mx[hr]);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            alpha[hr] = fast_exp2(m_run[hr] - m_use);
            m_run[hr] = m_new;
            mx[hr] = m_use;
            l_run[hr] *= alpha[hr];
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float pe = fast_exp2(s[nt][e] - mx[e >> 1]);
                s[nt][e] = pe;
                l_run[e >> 1] += pe;
            }
        }
#pragma unroll
        for (int i = 0; i < NT; ++i) {
            o[i][0] *= alpha[0];
            o[i][1] *= alpha[0];
            o[i][2] *= alpha[1];
            o[i][3] *= alpha[1];
        }
        // O += P V
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t a0 = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
            const uint32_t a1 = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
            const uint32_t a2 = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            const uint32_t a3 = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            const int key = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int n = 0; n < NT; n += 2) {
                uint32_t b0, b1, b2, b3;
                ldmatrix_x4_trans(smem_u32(sV + swz<CH>(key, n + (lane >> 4))), b0, b1, b2, b3);
                mma_bf16_16816(o[n], a0, a1, a2, a3, b0, b1);
                mma_bf16_16816(o[n + 1], a0, a1, a2, a3, b2, b3);
            }
        }
    }
    cp_async_wait<0>();

    // ---- epilogue
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 1);
        l_run[hr] += __shfl_xor_sync(0xffffffffu, l_run[hr], 2);
    }
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int r = warp * 16 + g_lane + hr * 8;
        const int tk = tok0 + r / G;
        if (tk >= n_rows_tok) continue;
        const int h = kvh * G + (r % G);
        const float inv = l_run[hr] > 0.f ? 1.f / l_run[hr] : 0.f;
        const float lse2 = m_run[hr] + log2f(l_run[hr]);
        if constexpr (MODE == MQMode::kExtend) {
            const int64_t row = (int64_t)(qo0 + tk) * p.q_heads + h;
            __nv_bfloat16* dst = p.out + row * D;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int c = n * 8 + 2 * t_lane;
                *reinterpret_cast<uint32_t*>(dst + c) = pack_bf16(o[n][2 * hr] * inv, o[n][2 * hr + 1] * inv);
            }
            if (p.lse && t_lane == 0) p.lse[row] = lse2 * kLn2;
        } else {
            const int64_t row = ((int64_t)(qo0 + tk) * p.q_heads + h) * p.seg_chunks + (z % p.seg_chunks);
            float* dst = p.part_o + row * D;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                const int c = n * 8 + 2 * t_lane;
                *reinterpret_cast<float2*>(dst + c) = make_float2(o[n][2 * hr] * inv, o[n][2 * hr + 1] * inv);
            }
            if (t_lane == 0) p.part_lse[row] = lse2;
        }
    }
}

}  // namespace rc
