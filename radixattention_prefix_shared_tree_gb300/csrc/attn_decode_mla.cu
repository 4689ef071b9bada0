// attn_decode for the latent (multi-head latent attention) layout: one KV
// head whose 576-wide row is the key (512 latent + 64 rotary columns) and
// whose first 512 columns are the value, read by 128 query heads.  The SGLang
// engineering article (section 1, MLA) notes that with a single KV head the
// decode kernel should serve several query heads per block to cut KV traffic;
// here a CTA serves 16 heads and the 8 head blocks of a request share every K
// row through L2.
//
// CTA = (key chunk, 16-head block, request), 4 warps, 32-key tiles gathered
// by slot with cp.async (slot ids travel through the pipeline two tiles ahead
// of the rows that need them).  Per tile: warp w computes S for keys
// 8w..8w+7 against the 16 heads (36 k-steps of mma.sync over 576 columns),
// the four warps agree on the running max through shared memory, P goes to
// shared memory as bf16, and warp w accumulates O for output columns
// 128w..128w+127 (P.V over the tile's 32 keys).  Output: the final bf16 row
// when one chunk covers the request, else normalised partials for the merge.

#include "attn_decode_mla_tc.cuh"
#include "common.cuh"

namespace rc_mla {

constexpr int DK = 576, DV = 512;
constexpr int HB = 16;          // heads per CTA
constexpr int TK = 32;          // keys per tile
constexpr int STAGES = 2;
constexpr int RING = 4;         // slot-id tiles in flight
constexpr int CHK = DK / 8;     // 72 chunks of 16 bytes per row
constexpr int PSTRIDE = 80;     // bytes per P row (32 bf16 + pad: conflict-free ldmatrix)
constexpr int TILE_BYTES = TK * DK * 2;

__host__ __device__ constexpr int smem_bytes() {
    return HB * DK * 2 + STAGES * TILE_BYTES + HB * PSTRIDE + RING * TK * 4 + 2 * 4 * HB * 4;
}

struct Params {
    const __nv_bfloat16* q;      // [B][Hq][576]
    const __nv_bfloat16* pool;   // [n_slots][576]
    int64_t n_slots;
    int32_t q_heads;
    float scale_log2;
    int32_t* err;
    const int32_t* table;
    const int32_t* start;
    const int32_t* len;
    int64_t table_len;
    int32_t chunk, n_chunks;
    float* part_o;               // [B][Hq][n_chunks][512]
    float* part_lse;             // [B][Hq][n_chunks]
    __nv_bfloat16* out;          // [B][Hq][512] (single chunk)
    float* lse;                  // [B][Hq] or NULL (single chunk)
};

template <bool FUSED>
__global__ void __launch_bounds__(128, 2) mla_decode_kernel(const Params p) {
    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* sQ = smem;                                  // [16][576] swizzled
    unsigned char* sKV = sQ + HB * DK * 2;                     // STAGES x [32][576]
    unsigned char* sP = sKV + STAGES * TILE_BYTES;             // [16][PSTRIDE]
    int32_t* sSlot = reinterpret_cast<int32_t*>(sP + HB * PSTRIDE);  // [RING][32]
    float* sMax = reinterpret_cast<float*>(sSlot + RING * TK);  // [4][16]
    float* sSum = sMax + 4 * HB;                                // [4][16]

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g_lane = lane >> 2, t_lane = lane & 3;
    const int chunk = blockIdx.x, hb = blockIdx.y, b = blockIdx.z;
    const int64_t row0 = p.start[b];
    int L = p.len[b];
    if (row0 < 0 || L < 0 || row0 + L > p.table_len) {
        if (tid == 0 && hb == 0 && chunk == 0) rc::flag_error(p.err, rc::kErrBadSlot);
        L = 0;
    }
    if (FUSED && tid == 0 && hb == 0 && L > p.chunk) rc::flag_error(p.err, rc::kErrBadSlot);
    const int k0 = chunk * p.chunk;
    const int count = max(0, min(L - k0, p.chunk));
    if (!FUSED && count == 0) return;
    const int32_t* keys = p.table + row0 + k0;
    const int n_tiles = (count + TK - 1) / TK;

    auto copy_slots = [&](int t) {
        if (tid < TK) {
            const int key = t * TK + tid;
            const bool ok = t < n_tiles && key < count;
            rc::cp_async4(rc::smem_u32(sSlot + (t % RING) * TK + tid), ok ? keys + key : keys, ok ? 4u : 0u);
        }
    };
    auto issue = [&](int t) {
        if (t >= n_tiles) return;
        unsigned char* sK = sKV + (t % STAGES) * TILE_BYTES;
        const int32_t* ring = sSlot + (t % RING) * TK;
        for (int i = tid; i < TK * CHK; i += 128) {
            const int r = i / CHK, c = i % CHK;
            int slot = ring[r];
            uint32_t bytes = 16;
            if (t * TK + r >= count) { slot = 0; bytes = 0; }
            else if (slot < 0 || (int64_t)slot >= p.n_slots) {
                rc::flag_error(p.err, rc::kErrBadSlot);
                slot = 0;
                bytes = 0;
            }
            rc::cp_async16(rc::smem_u32(sK + rc::swz<CHK>(r, c)), p.pool + (int64_t)slot * DK + c * 8, bytes);
        }
    };

    // prologue: slot ids of tiles 0..2; then Q + tile 0
#pragma unroll
    for (int t = 0; t < 3; ++t) copy_slots(t);
    rc::cp_async_commit();
    rc::cp_async_wait<0>();
    __syncthreads();
    for (int i = tid; i < HB * CHK; i += 128) {
        const int r = i / CHK, c = i % CHK;
        rc::cp_async16(rc::smem_u32(sQ + rc::swz<CHK>(r, c)),
                       p.q + ((int64_t)b * p.q_heads + hb * HB + r) * DK + c * 8, 16u);
    }
    issue(0);
    rc::cp_async_commit();

    float o[16][4];  // O for heads g, g+8 x this warp's 128 output columns
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    // group committed at iteration t holds K of tile t+1 and slot ids of tile t+3
    for (int t = 0; t < n_tiles; ++t) {
        rc::cp_async_wait<0>();
        __syncthreads();
        issue(t + 1);
        copy_slots(t + 3);
        rc::cp_async_commit();
        const unsigned char* sK = sKV + (t % STAGES) * TILE_BYTES;

        // S (16 heads x 8 keys of this warp) over 576 columns
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const int qr = (lane & 7) + ((lane >> 3) & 1) * 8;
            const int kr = warp * 8 + (lane & 7);
#pragma unroll 4
            for (int ks = 0; ks < DK / 16; ks += 2) {
                uint32_t b0, b1, b2, b3;
                rc::ldmatrix_x4(rc::smem_u32(sK + rc::swz<CHK>(kr, ks * 2 + (lane >> 3))), b0, b1, b2, b3);
                uint32_t a0, a1, a2, a3;
                rc::ldmatrix_x4(rc::smem_u32(sQ + rc::swz<CHK>(qr, ks * 2 + (lane >> 4))), a0, a1, a2, a3);
                rc::mma_bf16_16816(s, a0, a1, a2, a3, b0, b1);
                rc::ldmatrix_x4(rc::smem_u32(sQ + rc::swz<CHK>(qr, (ks + 1) * 2 + (lane >> 4))), a0, a1, a2, a3);
                rc::mma_bf16_16816(s, a0, a1, a2, a3, b2, b3);
            }
        }
        // s[0], s[1]: head g, keys 2t, 2t+1; s[2], s[3]: head g+8
        const int kbase = t * TK + warp * 8 + 2 * t_lane;
        const bool v0 = kbase < count, v1 = kbase + 1 < count;
        s[0] = v0 ? s[0] * p.scale_log2 : -INFINITY;
        s[1] = v1 ? s[1] * p.scale_log2 : -INFINITY;
        s[2] = v0 ? s[2] * p.scale_log2 : -INFINITY;
        s[3] = v1 ? s[3] * p.scale_log2 : -INFINITY;
        float mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]);
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        if (t_lane == 0) {
            sMax[warp * HB + g_lane] = mx0;
            sMax[warp * HB + g_lane + 8] = mx1;
        }
        __syncthreads();
        float tm0 = sMax[g_lane], tm1 = sMax[g_lane + 8];
#pragma unroll
        for (int w = 1; w < 4; ++w) {
            tm0 = fmaxf(tm0, sMax[w * HB + g_lane]);
            tm1 = fmaxf(tm1, sMax[w * HB + g_lane + 8]);
        }
        const float mn0 = fmaxf(m_run[0], tm0), mn1 = fmaxf(m_run[1], tm1);
        const float mu0 = mn0 == -INFINITY ? 0.f : mn0, mu1 = mn1 == -INFINITY ? 0.f : mn1;
        const float al0 = rc::fast_exp2(m_run[0] - mu0), al1 = rc::fast_exp2(m_run[1] - mu1);
        m_run[0] = mn0;
        m_run[1] = mn1;
        const float p0 = rc::fast_exp2(s[0] - mu0), p1 = rc::fast_exp2(s[1] - mu0);
        const float p2 = rc::fast_exp2(s[2] - mu1), p3 = rc::fast_exp2(s[3] - mu1);
        // P to shared memory: row = head, column = key within the tile
        *reinterpret_cast<uint32_t*>(sP + g_lane * PSTRIDE + (warp * 8 + 2 * t_lane) * 2) = rc::pack_bf16(p0, p1);
        *reinterpret_cast<uint32_t*>(sP + (g_lane + 8) * PSTRIDE + (warp * 8 + 2 * t_lane) * 2) =
            rc::pack_bf16(p2, p3);
        float ps0 = p0 + p1, ps1 = p2 + p3;
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 1);
        ps0 += __shfl_xor_sync(0xffffffffu, ps0, 2);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 1);
        ps1 += __shfl_xor_sync(0xffffffffu, ps1, 2);
        if (t_lane == 0) {
            sSum[warp * HB + g_lane] = ps0;
            sSum[warp * HB + g_lane + 8] = ps1;
        }
        __syncthreads();
        l_run[0] = l_run[0] * al0 + sSum[g_lane] + sSum[HB + g_lane] + sSum[2 * HB + g_lane] + sSum[3 * HB + g_lane];
        l_run[1] = l_run[1] * al1 + sSum[g_lane + 8] + sSum[HB + g_lane + 8] + sSum[2 * HB + g_lane + 8] +
                   sSum[3 * HB + g_lane + 8];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            o[i][0] *= al0;
            o[i][1] *= al0;
            o[i][2] *= al1;
            o[i][3] *= al1;
        }
        // O (16 heads x 128 columns of this warp) += P (16 x 32) V (32 x 128)
#pragma unroll
        for (int kk = 0; kk < TK / 16; ++kk) {
            uint32_t a0, a1, a2, a3;
            {
                const int pr = (lane & 7) + ((lane >> 3) & 1) * 8;
                const int pc = kk * 2 + (lane >> 4);
                rc::ldmatrix_x4(rc::smem_u32(sP + pr * PSTRIDE + pc * 16), a0, a1, a2, a3);
            }
            const int vr = kk * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int n = 0; n < 16; n += 2) {
                uint32_t b0, b1, b2, b3;
                rc::ldmatrix_x4_trans(rc::smem_u32(sK + rc::swz<CHK>(vr, warp * 16 + n + (lane >> 4))), b0, b1, b2,
                                      b3);
                rc::mma_bf16_16816(o[n], a0, a1, a2, a3, b0, b1);
                rc::mma_bf16_16816(o[n + 1], a0, a1, a2, a3, b2, b3);
            }
        }
    }
    rc::cp_async_wait<0>();

    const float inv0 = l_run[0] > 0.f ? 1.f / l_run[0] : 0.f;
    const float inv1 = l_run[1] > 0.f ? 1.f / l_run[1] : 0.f;
    const float lse0 = l_run[0] > 0.f ? m_run[0] + log2f(l_run[0]) : -INFINITY;
    const float lse1 = l_run[1] > 0.f ? m_run[1] + log2f(l_run[1]) : -INFINITY;
#pragma unroll
    for (int hr = 0; hr < 2; ++hr) {
        const int head = hb * HB + g_lane + 8 * hr;
        const float inv = hr ? inv1 : inv0;
        if (FUSED) {
            __nv_bfloat16* dst = p.out + ((int64_t)b * p.q_heads + head) * DV + warp * 128;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                *reinterpret_cast<uint32_t*>(dst + n * 8 + 2 * t_lane) =
                    rc::pack_bf16(o[n][2 * hr] * inv, o[n][2 * hr + 1] * inv);
            if (p.lse && warp == 0 && t_lane == 0)
                p.lse[(int64_t)b * p.q_heads + head] = (hr ? lse1 : lse0) * rc::kLn2;
        } else {
            const int64_t idx = ((int64_t)b * p.q_heads + head) * p.n_chunks + chunk;
            float* dst = p.part_o + idx * DV + warp * 128;
#pragma unroll
            for (int n = 0; n < 16; ++n)
                *reinterpret_cast<float2*>(dst + n * 8 + 2 * t_lane) =
                    make_float2(o[n][2 * hr] * inv, o[n][2 * hr + 1] * inv);
            if (warp == 0 && t_lane == 0) p.part_lse[idx] = hr ? lse1 : lse0;
        }
    }
}

// LSE merge of the chunk partials, one warp per (request, head).
__global__ void __launch_bounds__(32) mla_merge_kernel(const Params p) {
    constexpr int PER = DV / 32;
    const int bh = blockIdx.x;
    const int b = bh / p.q_heads;
    const int lane = threadIdx.x;
    const int64_t row0 = p.start[b];
    const int L = p.len[b];
    // a row the split pass rejected (outside the table) wrote no partials
    int nc = (row0 < 0 || L < 0 || row0 + L > p.table_len) ? 0 : (L + p.chunk - 1) / p.chunk;
    if (nc > p.n_chunks) {
        if (lane == 0 && bh % p.q_heads == 0) rc::flag_error(p.err, rc::kErrBadSlot);
        nc = p.n_chunks;
    }
    // a split kernel that gave up on a bounded wait (or met the flag of an
    // earlier one) left its partials unwritten: use none of them
    if (p.err && (*reinterpret_cast<volatile int32_t*>(p.err) & rc::kErrTimeout)) nc = 0;
    float m = -INFINITY;
    for (int c = 0; c < nc; ++c) m = fmaxf(m, p.part_lse[(int64_t)bh * p.n_chunks + c]);
    float acc[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) acc[j] = 0.f;
    float w = 0.f;
    for (int c = 0; c < nc; ++c) {
        const int64_t row = (int64_t)bh * p.n_chunks + c;
        const float l2 = p.part_lse[row];
        if (l2 == -INFINITY) continue;
        const float e = rc::fast_exp2(l2 - m);
        w += e;
#pragma unroll
        for (int j = 0; j < PER; ++j) acc[j] += e * p.part_o[row * DV + lane + 32 * j];
    }
    const float inv = w > 0.f ? 1.f / w : 0.f;
#pragma unroll
    for (int j = 0; j < PER; ++j) p.out[(int64_t)bh * DV + lane + 32 * j] = __float2bfloat16_rn(acc[j] * inv);
    if (p.lse && lane == 0) p.lse[bh] = w > 0.f ? (m + log2f(w)) * rc::kLn2 : -INFINITY;
}

}  // namespace rc_mla

namespace rc_host {

// 128 query heads: the tcgen05 kernel (attn_decode_mla_tc.cuh), all heads in
// one CTA per (key chunk, value half, request).
bool mla_use_tc(int32_t q_heads) { return q_heads == rc_mla_tc::M; }

// Plan of the latent decode: keys per CTA and chunks per request.
void mla_plan(int32_t batch, int32_t q_heads, int32_t max_len, int* chunk, int* n_chunks) {
    const int64_t sms = sm_count();
    if (mla_use_tc(q_heads)) {
        // about four CTAs per SM over the batch (rows are about half the
        // longest on average, two value halves per chunk), 256..4096 keys
        int64_t c = max_len > 0 ? (int64_t)batch * max_len / (4 * sms) : rc_mla_tc::TN;
        c = (c + rc_mla_tc::TN - 1) / rc_mla_tc::TN * rc_mla_tc::TN;
        if (c < 256) c = 256;
        if (c > 4096) c = 4096;
        *chunk = (int)c;
        *n_chunks = max_len > 0 ? (int)((max_len + c - 1) / c) : 1;
        return;
    }
    const int64_t base = (int64_t)batch * (q_heads / rc_mla::HB);
    int64_t splits = base > 0 ? (4 * sms + base - 1) / base : 1;
    const int64_t max_splits = max_len > 0 ? (max_len + 1023) / 1024 : 1;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    int64_t c = max_len > 0 ? (max_len + splits - 1) / splits : rc_mla::TK;
    c = (c + rc_mla::TK - 1) / rc_mla::TK * rc_mla::TK;
    *chunk = (int)c;
    *n_chunks = max_len > 0 ? (int)((max_len + c - 1) / c) : 1;
}

size_t mla_workspace(int32_t batch, int32_t q_heads, int32_t max_len) {
    int chunk = 0, nc = 0;
    mla_plan(batch, q_heads, max_len, &chunk, &nc);
    if (nc <= 1) return 256;
    const size_t rows = (size_t)batch * q_heads * nc;
    const size_t a = (rows * rc_mla::DV * sizeof(float) + 255) & ~size_t(255);
    return a + ((rows * sizeof(float) + 255) & ~size_t(255));
}

rc_status mla_decode(const rc_attn_desc* desc, const void* q, const rc_kv_table* kv, int32_t batch, void* out,
                     float* lse, void* ws, size_t ws_bytes, cudaStream_t st) {
    const rc_pool_desc& P = desc->pool;
    if (P.kv_heads != 1 || P.head_dim_k != rc_mla::DK || P.head_dim_v != rc_mla::DV) return RC_ERR_UNSUPPORTED;
    if (desc->q_heads % rc_mla::HB) return RC_ERR_UNSUPPORTED;
    if (ws_bytes < mla_workspace(batch, desc->q_heads, kv->max_len)) return RC_ERR_ARG;
    rc_mla::Params p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.pool = static_cast<const __nv_bfloat16*>(P.k);
    p.n_slots = P.n_slots;
    p.q_heads = desc->q_heads;
    p.scale_log2 = desc->sm_scale * rc::kLog2e;
    p.err = P.err;
    p.table = kv->slots;
    p.start = kv->start;
    p.len = kv->len;
    p.table_len = kv->table_len;
    mla_plan(batch, desc->q_heads, kv->max_len, &p.chunk, &p.n_chunks);
    const size_t rows = (size_t)batch * desc->q_heads * p.n_chunks;
    p.part_o = static_cast<float*>(ws);
    p.part_lse = reinterpret_cast<float*>(static_cast<unsigned char*>(ws) +
                                          ((rows * rc_mla::DV * sizeof(float) + 255) & ~size_t(255)));
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    cudaError_t e;
    if (mla_use_tc(desc->q_heads)) {
        rc_mla_tc::Params t{};
        t.q = p.q;
        t.pool = p.pool;
        t.n_slots = p.n_slots;
        t.scale_log2 = p.scale_log2;
        t.err = p.err;
        t.table = p.table;
        t.start = p.start;
        t.len = p.len;
        t.table_len = p.table_len;
        t.chunk = p.chunk;
        t.n_chunks = p.n_chunks;
        t.part_o = p.part_o;
        t.part_lse = p.part_lse;
        t.out = p.out;
        t.lse = p.lse;
        if (p.n_chunks == 1) return launch_status(rc_mla_tc::launch<true>(t, p.n_chunks, batch, st));
        if (rc_mla_tc::launch<false>(t, p.n_chunks, batch, st) != cudaSuccess) return RC_ERR_CUDA;
        rc_mla::mla_merge_kernel<<<(unsigned)(batch * desc->q_heads), 32, 0, st>>>(p);
        return launch_status(cudaGetLastError());
    }
    constexpr int smem = rc_mla::smem_bytes();
    dim3 grid(p.n_chunks, desc->q_heads / rc_mla::HB, batch);
    if (p.n_chunks == 1) {
        e = ensure_smem<rc_mla::mla_decode_kernel<true>>(smem);
        if (e != cudaSuccess) return RC_ERR_CUDA;
        rc_mla::mla_decode_kernel<true><<<grid, 128, smem, st>>>(p);
    } else {
        e = ensure_smem<rc_mla::mla_decode_kernel<false>>(smem);
        if (e != cudaSuccess) return RC_ERR_CUDA;
        rc_mla::mla_decode_kernel<false><<<grid, 128, smem, st>>>(p);
        if (cudaGetLastError() != cudaSuccess) return RC_ERR_CUDA;
        rc_mla::mla_merge_kernel<<<(unsigned)(batch * desc->q_heads), 32, 0, st>>>(p);
    }
    return launch_status(cudaGetLastError());
}

}  // namespace rc_host
