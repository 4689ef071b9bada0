// attn_decode: one new token per request attends to its whole cached context,
// read through the request's slot table (decode phase of the SageMaker LMI
// article; the K/V come from the radix-tree cache of inference-notes note 49,
// section 2).  Memory-bound: every K/V row of the context is read once per KV
// head per step, so the design goal is to stream rows at HBM speed.
//
//  1. cascade pass (when the batch shares prefixes): each shared segment is
//     read once for all rows below it by the tcgen05 many-row kernel
//     (attn_tc2.cuh), one partial per (row, head, segment, key chunk).
//  2. table pass: one warp per item (request, KV head[, key chunk]).  The G
//     query heads of the KV head share each K/V row (grouped-query head
//     grouping).  Each warp gathers its keys by slot with 16-byte cp.async
//     into its own two-stage ring of 16-key tiles; the products run on
//     mma.sync with the keys on the M side and the G heads on the N side (so
//     G = 4 or 8 wastes at most half of an n8 tile instead of 12 of 16 rows),
//     and P moves from accumulator to operand layout with movmatrix.  With
//     one chunk per row the warp's epilogue folds in the row's cascade
//     partials and writes the output (fused); otherwise it writes a
//     normalised partial and its log-sum-exp per (request, head, chunk).
//  3. merge pass (split rows only): per (request, head), combine all
//     partials by log-sum-exp.

#include "attn_tc2.cuh"
#include "common.cuh"

namespace {

constexpr int kDecKeys = 64;    // chunk sizes are multiples of this

struct DecParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* pool_k;
    const __nv_bfloat16* pool_v;
    int64_t n_slots;
    int32_t kv_heads, q_heads;
    float scale_log2;
    int32_t* err;
    const int32_t* table;
    const int32_t* start;
    const int32_t* len;
    int64_t table_len;
    int32_t chunk;       // keys per CTA
    int32_t n_chunks;    // max chunks per request (partial stride)
    float* part_o;       // [B][Hq][n_chunks][D]      (unfused)
    float* part_lse;     // [B][Hq][n_chunks]
    // fused epilogue: combine with the cascade partials and write the result
    const float* seg_o;  // [total_seg_rows][Hq][seg_chunks][D]
    const float* seg_lse;
    const int32_t* req_seg_indptr;  // NULL: no cascade
    const int32_t* req_seg_pos;
    int32_t seg_chunks;
    __nv_bfloat16* out;
    float* lse;
    // attn_decode_append: each row's last key comes from here and is stored
    const __nv_bfloat16* k_new;  // [B][kv_heads][D] or NULL
    const __nv_bfloat16* v_new;
    // FP8 pool: pool_k / pool_v hold E4M3 codes, these the per-row scales
    const float* k_scale;  // [n_slots][kv_heads]
    const float* v_scale;
};

// Decode with one warp per item (request b, KV head, key chunk).  Each warp
// streams its keys through a private ring of 16-key tiles (one m16 tile of
// the swapped product) with cp.async, synchronising with __syncwarp only, so
// the warps of an SM overlap each other's load latency and epilogues freely.
// Wait until the grid this one depends on programmatically (the cascade
// kernel) has finished and its writes are visible; returns at once when the
// grid was launched without that dependency.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }

constexpr int kWarpKeys = 16;
constexpr int kWarpsPerCta = 14;  // one CTA per SM (14 x 16 KB + the CTA's 1 KB reserve fit; seven CTAs of
constexpr int kCtasPerSm = 1;     // two warps would not): 2128 resident warps, the 2048 (row, KV head) items
                                  // of a 256-row GQA-8 batch in one wave

// Per-warp ring: S stages of one 16-key tile each (K then V, then for an FP8
// pool the tile's 16 K scales and 16 V scales); a stage is refilled as soon
// as its tile is reduced, so S tiles are in flight while the warp waits.
template <bool FP8>
__host__ __device__ constexpr int warp_stages() { return FP8 ? 3 : 2; }
template <int D, bool FP8>
__host__ __device__ constexpr int tile_bytes() { return kWarpKeys * D * (FP8 ? 1 : 2); }
template <int D, bool FP8>
__host__ __device__ constexpr int stage_bytes() { return 2 * tile_bytes<D, FP8>() + (FP8 ? 2 * kWarpKeys * 4 : 0); }
template <int D, bool FP8>
__host__ __device__ constexpr int warp_smem_bytes() {  // the K/V ring only (Q and slot ids in registers)
    return warp_stages<FP8>() * stage_bytes<D, FP8>();
}
template <int D, bool FP8>
__host__ __device__ constexpr int dec_smem_bytes() {
    return kWarpsPerCta * warp_smem_bytes<D, FP8>();
}

template <int D, int G, bool FUSED, bool FP8>
__global__ void __launch_bounds__(32 * kWarpsPerCta, kCtasPerSm) decode_split_kernel(const DecParams p, int n_items) {
    constexpr int ESZ = FP8 ? 1 : 2;                // bytes per K/V element
    constexpr int CH = D * ESZ / 16;                // 16-byte chunks per row
    constexpr int KS = D / 16;
    constexpr int PER = kWarpKeys * CH / 32;        // chunks per lane per matrix
    constexpr int S = warp_stages<FP8>();
    constexpr int TILE_BYTES = tile_bytes<D, FP8>();
    constexpr int STAGE_BYTES = stage_bytes<D, FP8>();
    static_assert(kWarpKeys == 16, "slot ids: one lane per key");
    static_assert(!FP8 || D == 128, "FP8 pools: head_dim 128");
    // the epilogue reuses the ring: [8][D] fp32 outputs plus the merge scratch
    static_assert(warp_smem_bytes<D, FP8>() >= 8 * D * 4 + 32 + 32 * 8 + G * 32 * 4 + G * 8, "epilogue scratch");
    extern __shared__ __align__(128) unsigned char smem[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g_lane = lane >> 2, t_lane = lane & 3;
    // the next step's cascade kernel (launched as this grid's dependent) may
    // take SMs as they free up: it waits for this grid's end itself
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    const int it = blockIdx.x * kWarpsPerCta + warp;
    if (it >= n_items) {
        grid_dep_wait();
        return;
    }
    unsigned char* wbase = smem + warp * warp_smem_bytes<D, FP8>();

    const int kvh = it % p.kv_heads;
    const int rest = it / p.kv_heads;
    const int chunk = rest % p.n_chunks;
    const int b = rest / p.n_chunks;
    const int64_t row0 = p.start[b];
    int L = p.len[b];
    if (row0 < 0 || L < 0 || row0 + L > p.table_len) {  // row outside the table: read nothing
        if (lane == 0 && kvh == 0 && chunk == 0) rc::flag_error(p.err, rc::kErrBadSlot);
        L = 0;
    }
    if (FUSED && lane == 0 && kvh == 0 && L > p.chunk) rc::flag_error(p.err, rc::kErrBadSlot);
    const int k0 = chunk * p.chunk;
    const int count = max(0, min(L - k0, p.chunk));
    if (!FUSED && count == 0) {
        grid_dep_wait();
        return;
    }
    const int32_t* keys = p.table + row0 + k0;
    const int n_tiles = (count + kWarpKeys - 1) / kWarpKeys;
    // fused epilogue: the cascade partials this row folds in; the row offsets
    // of the first 32 (lane j: partial j) are read now, ahead of the main loop
    // (the segment tables are the caller's inputs, not the cascade's output)
    int e0 = 0, n_parts = 0;
    if (FUSED && p.req_seg_indptr) {
        e0 = p.req_seg_indptr[b];
        n_parts = (p.req_seg_indptr[b + 1] - e0) * p.seg_chunks;
    }
    auto part_row = [&](int j) -> int64_t {
        return j < n_parts ? (int64_t)p.req_seg_pos[e0 + j / p.seg_chunks] * p.q_heads * p.seg_chunks +
                                 (j % p.seg_chunks)
                           : 0;
    };
    const int64_t first_row = part_row(lane);
    // attn_decode_append: the row's last key (position L-1) is the step's new
    // token.  The warp whose keys hold it gathers it from k_new/v_new and
    // writes it to its pool slot (lanes 0..CH-1 the K row, CH..2CH-1 the V row).
    const int new_at = (!FP8 && p.k_new && L > 0 && L - 1 >= k0 && L - 1 < k0 + count) ? L - 1 - k0 : -1;
    if (new_at >= 0) {
        const int slot = keys[new_at];
        if (slot < 0 || (int64_t)slot >= p.n_slots) {
            if (lane == 0) rc::flag_error(p.err, rc::kErrBadSlot);
        } else if (lane < 2 * CH) {
            const int c = lane % CH;
            const int64_t off = ((int64_t)slot * p.kv_heads + kvh) * D + c * 8;
            const int64_t src = ((int64_t)b * p.kv_heads + kvh) * D + c * 8;
            if (lane < CH)
                *reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(p.pool_k) + off) =
                    *reinterpret_cast<const uint4*>(p.k_new + src);
            else
                *reinterpret_cast<uint4*>(const_cast<__nv_bfloat16*>(p.pool_v) + off) =
                    *reinterpret_cast<const uint4*>(p.v_new + src);
        }
    }

    // Slot ids are prefetched into registers one tile ahead: lane l (and
    // l + 16) holds the slot of key l of a tile.
    auto slot_of = [&](int t) -> int {
        const int key = t * kWarpKeys + (lane & 15);
        return (t < n_tiles && key < count) ? __ldg(keys + key) : 0;
    };
    // a request's own keys are read once per step: they should not push the
    // shared prefix (read by the cascade kernel every step) out of L2
    const uint64_t pol = rc::l2_policy_evict_first();
    auto issue = [&](int t, int tslots) {
        if (t < n_tiles) {
            unsigned char* sK = wbase + (t % S) * STAGE_BYTES;
            unsigned char* sV = sK + TILE_BYTES;
#pragma unroll
            for (int i = 0; i < PER; ++i) {
                const int lin = i * 32 + lane;
                const int r = lin / CH, c = lin % CH;
                const int slot = __shfl_sync(0xffffffffu, tslots, r);
                uint32_t bytes = 16;
                const unsigned char* bk = reinterpret_cast<const unsigned char*>(p.pool_k);
                const unsigned char* bv = reinterpret_cast<const unsigned char*>(p.pool_v);
                int64_t row = 0;
                if (t * kWarpKeys + r >= count) bytes = 0;
                else if (t * kWarpKeys + r == new_at) {  // the appended key, straight from its source
                    bk = reinterpret_cast<const unsigned char*>(p.k_new);
                    bv = reinterpret_cast<const unsigned char*>(p.v_new);
                    row = b;
                } else if (slot < 0 || (int64_t)slot >= p.n_slots) {
                    rc::flag_error(p.err, rc::kErrBadSlot);
                    bytes = 0;
                } else {
                    row = slot;
                }
                const int64_t roff = (row * p.kv_heads + kvh) * (D * ESZ) + c * 16;
                rc::cp_async16(rc::smem_u32(sK + rc::swz<CH>(r, c)), bk + roff, bytes, pol);
                rc::cp_async16(rc::smem_u32(sV + rc::swz<CH>(r, c)), bv + roff, bytes, pol);
            }
            if constexpr (FP8) {  // lanes 0-15: K scale of key lane, 16-31: V scale of key lane-16
                const int r = lane & 15;
                const bool ok = t * kWarpKeys + r < count && tslots >= 0 && (int64_t)tslots < p.n_slots;
                const float* src = (lane < 16 ? p.k_scale : p.v_scale) + (ok ? (int64_t)tslots * p.kv_heads + kvh : 0);
                rc::cp_async4(rc::smem_u32(sV + TILE_BYTES + lane * 4), src, ok ? 4u : 0u);
            }
        }
    };
    // prologue: slot ids of tiles 0 and 1, K/V of tile 0, and the Q operand
    // fragments straight from global memory (head g_lane of this KV head's
    // group, zero for g_lane >= G; two bf16 per register, as ldmatrix would
    // give them)
    // Tiles t..t+S-1 are in flight while the warp waits for tile t; tile
    // t+S goes into tile t's stage as soon as tile t has been reduced.
    int cur = slot_of(S), nxt;
#pragma unroll
    for (int i = 0; i < S; ++i) {
        issue(i, slot_of(i));
        rc::cp_async_commit();
    }
    uint32_t qb[KS][2];
    {
        const bool hv = g_lane < G;
        const uint32_t* qrow = reinterpret_cast<const uint32_t*>(
            p.q + ((int64_t)b * p.q_heads + kvh * G + (hv ? g_lane : 0)) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            if constexpr (FP8) {
                // f16 operands, and k-step ks takes dims 16ks+4t..16ks+4t+3 of
                // this lane's K words (see below): the same dims of Q
                qb[ks][0] = hv ? rc::bf16x2_to_f16x2(__ldg(qrow + ks * 8 + 2 * t_lane)) : 0u;
                qb[ks][1] = hv ? rc::bf16x2_to_f16x2(__ldg(qrow + ks * 8 + 2 * t_lane + 1)) : 0u;
            } else {
                qb[ks][0] = hv ? __ldg(qrow + ks * 8 + t_lane) : 0u;
                qb[ks][1] = hv ? __ldg(qrow + ks * 8 + 4 + t_lane) : 0u;
            }
        }
    }
    float o[KS][4];
#pragma unroll
    for (int i = 0; i < KS; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    for (int t = 0; t < n_tiles; ++t) {
        rc::cp_async_wait<S - 1>();  // tile t landed (later tiles may still be in flight)
        __syncwarp();
        nxt = slot_of(t + S + 1);
        const unsigned char* sK = wbase + (t % S) * STAGE_BYTES;
        const unsigned char* sV = sK + TILE_BYTES;
        const float* sSc = reinterpret_cast<const float*>(sV + TILE_BYTES);  // FP8: K scales, then V scales
        // S^T (16 keys x 8 heads) = K Q^T, even and odd k-steps in two
        // accumulators (two independent chains of MMAs)
        float s[4] = {0.f, 0.f, 0.f, 0.f};
        {
            float s2[4] = {0.f, 0.f, 0.f, 0.f};
            if constexpr (FP8) {
                // A fragment from E4M3 words: row g (and g+8), 16-byte chunk ks,
                // word t_lane = dims 16ks+4t..+3; the k-step's columns 2t, 2t+1
                // take the word's first two dims, 2t+8, 2t+9 the last two
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const uint32_t w0 = *reinterpret_cast<const uint32_t*>(sK + rc::swz<CH>(g_lane, ks) + 4 * t_lane);
                    const uint32_t w1 =
                        *reinterpret_cast<const uint32_t*>(sK + rc::swz<CH>(g_lane + 8, ks) + 4 * t_lane);
                    uint32_t a0, a1, a2, a3;
                    rc::e4m3x4_to_f16x4(w0, a0, a2);
                    rc::e4m3x4_to_f16x4(w1, a1, a3);
                    rc::mma_f16_16816(ks & 1 ? s2 : s, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                }
            } else {
                const int key = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    uint32_t a0, a1, a2, a3;
                    rc::ldmatrix_x4(rc::smem_u32(sK + rc::swz<CH>(key, ks * 2 + (lane >> 4))), a0, a1, a2, a3);
                    rc::mma_bf16_16816(ks & 1 ? s2 : s, a0, a1, a2, a3, qb[ks][0], qb[ks][1]);
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) s[i] += s2[i];
            if constexpr (FP8) {  // code products times the keys' scales
                const float k_lo = sSc[g_lane], k_hi = sSc[g_lane + 8];
                s[0] *= k_lo;
                s[1] *= k_lo;
                s[2] *= k_hi;
                s[3] *= k_hi;
            }
        }
        const int key_lo = t * kWarpKeys + g_lane;
        const bool v_lo = key_lo < count, v_hi = key_lo + 8 < count;
        s[0] = v_lo ? s[0] * p.scale_log2 : -INFINITY;
        s[1] = v_lo ? s[1] * p.scale_log2 : -INFINITY;
        s[2] = v_hi ? s[2] * p.scale_log2 : -INFINITY;
        s[3] = v_hi ? s[3] * p.scale_log2 : -INFINITY;
        // Online softmax with a lazy reference: exponentials are taken
        // against m_run, which moves (rescaling O and l) only when a head's
        // max grows past it by more than 2^8 -- the terms stay below 2^8, and
        // most tiles skip the 32 multiplies of the rescale.
        float mx[2] = {fmaxf(s[0], s[2]), fmaxf(s[1], s[3])};
        float alpha[2] = {1.f, 1.f};
        bool grow = false;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 4));
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 8));
            mx[j] = fmaxf(mx[j], __shfl_xor_sync(0xffffffffu, mx[j], 16));
            if (mx[j] > m_run[j] + 8.f) {
                alpha[j] = rc::fast_exp2(m_run[j] - mx[j]);  // 0 while nothing was seen
                m_run[j] = mx[j];
                grow = true;
            }
        }
        const float mu0 = m_run[0] == -INFINITY ? 0.f : m_run[0];
        const float mu1 = m_run[1] == -INFINITY ? 0.f : m_run[1];
        const float p0 = rc::fast_exp2(s[0] - mu0), p1 = rc::fast_exp2(s[1] - mu1);
        const float p2 = rc::fast_exp2(s[2] - mu0), p3 = rc::fast_exp2(s[3] - mu1);
        if (__any_sync(0xffffffffu, grow)) {
            l_run[0] *= alpha[0];
            l_run[1] *= alpha[1];
#pragma unroll
            for (int i = 0; i < KS; ++i) {
                o[i][0] *= alpha[0];
                o[i][1] *= alpha[1];
                o[i][2] *= alpha[0];
                o[i][3] *= alpha[1];
            }
        }
        l_run[0] += p0 + p2;
        l_run[1] += p1 + p3;
        if constexpr (FP8) {
            // P times the values' scales (f16), then O^T += V^T P^T with V^T
            // built from E4M3 bytes: this lane reads 16-byte chunk g of keys
            // 2t, 2t+1, 2t+8, 2t+9 (dims 16g..16g+15); product mt uses dims
            // 16g+2mt (row g) and 16g+2mt+1 (row g+8), paired across keys
            // with a byte permute
            const float v_lo = sSc[kWarpKeys + g_lane], v_hi = sSc[kWarpKeys + g_lane + 8];
            const uint32_t pb0 = rc::movmatrix_trans(rc::pack_f16(p0 * v_lo, p1 * v_lo));
            const uint32_t pb1 = rc::movmatrix_trans(rc::pack_f16(p2 * v_hi, p3 * v_hi));
            const uint4 w0 = *reinterpret_cast<const uint4*>(sV + rc::swz<CH>(2 * t_lane, g_lane));
            const uint4 w1 = *reinterpret_cast<const uint4*>(sV + rc::swz<CH>(2 * t_lane + 1, g_lane));
            const uint4 w8 = *reinterpret_cast<const uint4*>(sV + rc::swz<CH>(2 * t_lane + 8, g_lane));
            const uint4 w9 = *reinterpret_cast<const uint4*>(sV + rc::swz<CH>(2 * t_lane + 9, g_lane));
            const uint32_t x0[4] = {w0.x, w0.y, w0.z, w0.w}, x1[4] = {w1.x, w1.y, w1.z, w1.w};
            const uint32_t x8[4] = {w8.x, w8.y, w8.z, w8.w}, x9[4] = {w9.x, w9.y, w9.z, w9.w};
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;
                uint32_t a0, a1, a2, a3;
                rc::e4m3x4_to_f16x4(rc::prmt(x0[mt >> 1], x1[mt >> 1], sel), a0, a1);
                rc::e4m3x4_to_f16x4(rc::prmt(x8[mt >> 1], x9[mt >> 1], sel), a2, a3);
                rc::mma_f16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
            }
        } else {
            const uint32_t pb0 = rc::movmatrix_trans(rc::pack_bf16(p0, p1));
            const uint32_t pb1 = rc::movmatrix_trans(rc::pack_bf16(p2, p3));
            const int key = (lane & 7) + (lane >> 4) * 8;
#pragma unroll
            for (int mt = 0; mt < KS; ++mt) {
                uint32_t a0, a1, a2, a3;
                rc::ldmatrix_x4_trans(rc::smem_u32(sV + rc::swz<CH>(key, mt * 2 + ((lane >> 3) & 1))), a0, a1, a2,
                                      a3);
                rc::mma_bf16_16816(o[mt], a0, a1, a2, a3, pb0, pb1);
            }
        }
        __syncwarp();  // every lane has read tile t: its stage takes tile t+S
        issue(t + S, cur);
        rc::cp_async_commit();
        cur = nxt;
    }
    rc::cp_async_wait<0>();
    __syncwarp();

    // ---------------------------------------------------------- epilogue
#pragma unroll
    for (int j = 0; j < 2; ++j) {
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 4);
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 8);
        l_run[j] += __shfl_xor_sync(0xffffffffu, l_run[j], 16);
    }
    // this warp's normalised output per (head, dim) into its (now free) ring
    float* sE = reinterpret_cast<float*>(wbase);           // [8][D]
    float* sOwn = sE + 8 * D;                               // [8] log2-sum-exp per head
    const float inv0 = l_run[0] > 0.f ? 1.f / l_run[0] : 0.f;
    const float inv1 = l_run[1] > 0.f ? 1.f / l_run[1] : 0.f;
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
        // accumulator rows g and g+8 of product mt: dims d0 and d1
        const int d0 = FP8 ? 16 * g_lane + 2 * mt : mt * 16 + g_lane;
        const int d1 = FP8 ? d0 + 1 : d0 + 8;
        sE[(2 * t_lane) * D + d0] = o[mt][0] * inv0;
        sE[(2 * t_lane + 1) * D + d0] = o[mt][1] * inv1;
        sE[(2 * t_lane) * D + d1] = o[mt][2] * inv0;
        sE[(2 * t_lane + 1) * D + d1] = o[mt][3] * inv1;
    }
    if (g_lane == 0) {
        sOwn[2 * t_lane] = l_run[0] > 0.f ? m_run[0] + log2f(l_run[0]) : -INFINITY;
        sOwn[2 * t_lane + 1] = l_run[1] > 0.f ? m_run[1] + log2f(l_run[1]) : -INFINITY;
    }
    __syncwarp();
    // The cascade kernel, when there is one, may still be running (this
    // grid is its programmatic dependent): wait for it before reading its
    // partials, and in any case before leaving, so that the end of this grid
    // implies the end of both.
    grid_dep_wait();
    if constexpr (!FUSED) {
        for (int h = 0; h < G; ++h) {
            const int64_t idx = ((int64_t)b * p.q_heads + kvh * G + h) * p.n_chunks + chunk;
            for (int d = lane; d < D; d += 32) p.part_o[idx * D + d] = sE[h * D + d];
            if (lane == 0) p.part_lse[idx] = sOwn[h];
        }
    } else {
        // the row's whole table part is here: fold in its cascade partials
        // (every chunk of every segment it reads; partial j of head h sits at
        // row part_row(j) + (kvh * G + h) * seg_chunks).  Partials come in
        // batches of 32: lane j loads partial j's G log-sum-exps in one
        // round, then every lane loads the batch's rows in a second round
        // (all independent loads), merged online against a running max.
        constexpr int kPB = 32;
        int64_t* sRow = reinterpret_cast<int64_t*>(sOwn + 8);   // [kPB]
        float* sL = reinterpret_cast<float*>(sRow + kPB);         // [G][kPB]
        const int sc = p.seg_chunks;
        float m_h[G], w_h[G], acc[G][D / 32];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            m_h[h] = sOwn[h];
            w_h[h] = sOwn[h] == -INFINITY ? 0.f : 1.f;
#pragma unroll
            for (int k = 0; k < D / 32; ++k) acc[h][k] = m_h[h] == -INFINITY ? 0.f : sE[h * D + lane + 32 * k];
        }
        // none after a cascade kernel gave up on a bounded wait (unwritten)
        const int n_use = (p.err && (*reinterpret_cast<volatile int32_t*>(p.err) & rc::kErrTimeout)) ? 0 : n_parts;
        for (int j0 = 0; j0 < n_use; j0 += kPB) {
            const int nb = min(kPB, n_use - j0);
            const int64_t my_row = j0 == 0 ? first_row : part_row(j0 + lane);
            if (lane < nb) {
                sRow[lane] = my_row;
#pragma unroll
                for (int h = 0; h < G; ++h) sL[h * kPB + lane] = p.seg_lse[my_row + (int64_t)(kvh * G + h) * sc];
            }
            __syncwarp();
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float mb = m_h[h];
                for (int j = 0; j < nb; ++j) mb = fmaxf(mb, sL[h * kPB + j]);
                if (mb == -INFINITY) continue;   // nothing yet for this head
                const float a = m_h[h] == -INFINITY ? 0.f : rc::fast_exp2(m_h[h] - mb);
                w_h[h] *= a;
#pragma unroll
                for (int k = 0; k < D / 32; ++k) acc[h][k] *= a;
                m_h[h] = mb;
            }
#pragma unroll 4
            for (int j = 0; j < nb; ++j) {
                const int64_t row = sRow[j];
#pragma unroll
                for (int h = 0; h < G; ++h) {
                    const float l2 = sL[h * kPB + j];
                    const float wj = l2 == -INFINITY ? 0.f : rc::fast_exp2(l2 - m_h[h]);
                    w_h[h] += wj;
                    const float* src = p.seg_o + (row + (int64_t)(kvh * G + h) * sc) * D + lane;
#pragma unroll
                    for (int k = 0; k < D / 32; ++k) {
                        const float v = src[32 * k];
                        acc[h][k] += wj == 0.f ? 0.f : wj * v;
                    }
                }
            }
            __syncwarp();
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const int64_t orow = (int64_t)b * p.q_heads + kvh * G + h;
            const float inv = w_h[h] > 0.f ? 1.f / w_h[h] : 0.f;
#pragma unroll
            for (int k = 0; k < D / 32; ++k)
                p.out[orow * D + lane + 32 * k] = __float2bfloat16_rn(acc[h][k] * inv);
            if (p.lse && lane == 0)
                p.lse[orow] = w_h[h] > 0.f ? (m_h[h] + log2f(w_h[h])) * rc::kLn2 : -INFINITY;
        }
    }
}

// Combine every partial of (request, head): cascade segments (all chunks)
// then the chunks of the request's own table row.
template <int D>
__global__ void __launch_bounds__(32) merge_kernel(const float* __restrict__ tail_o,
                                                   const float* __restrict__ tail_lse, int32_t n_chunks,
                                                   int32_t chunk, const int32_t* __restrict__ len,
                                                   const float* __restrict__ seg_o,
                                                   const float* __restrict__ seg_lse, int32_t seg_chunks,
                                                   const int32_t* __restrict__ req_seg_indptr,
                                                   const int32_t* __restrict__ req_seg_pos, int32_t q_heads,
                                                   const int32_t* __restrict__ start, int64_t table_len,
                                                   __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                                   int32_t* err) {
    constexpr int PER = D / 32;
    const int bh = blockIdx.x;
    const int b = bh / q_heads, h = bh % q_heads;
    const int lane = threadIdx.x;
    // launched as the split pass's programmatic dependent: let the next
    // kernel launch, then wait for the split pass (and through it the
    // cascade) before reading anything they wrote
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
    grid_dep_wait();
    const int64_t row0 = start[b];
    const int L = len[b];
    // a row the split pass rejected (outside the table) wrote no partials
    int nc = (row0 < 0 || L < 0 || row0 + L > table_len) ? 0 : (L + chunk - 1) / chunk;
    if (nc > n_chunks) {  // len[b] above the caller's max_len: the split pass skipped keys
        if (lane == 0 && h == 0) rc::flag_error(err, rc::kErrBadSlot);
        nc = n_chunks;
    }
    // a cascade kernel that gave up on a bounded wait (or met the flag of an
    // earlier one) left its partials unwritten: use none of them
    const bool casc_ok = !(err && (*reinterpret_cast<volatile int32_t*>(err) & rc::kErrTimeout));
    const int s0 = req_seg_indptr && casc_ok ? req_seg_indptr[b] : 0;
    const int ns = req_seg_indptr && casc_ok ? req_seg_indptr[b + 1] - s0 : 0;
    // partials j < ns * seg_chunks: cascade (segment entry j / seg_chunks,
    // chunk j % seg_chunks); then the nc chunks of the row's own table part.
    // Batches of 32: lane j loads partial j's log-sum-exp (one round), then
    // every lane reads the batch's rows (independent loads), merged online.
    const int n_all = ns * seg_chunks + nc;
    __shared__ float sL[32];
    __shared__ const float* sSrc[32];
    float m = -INFINITY, wsum = 0.f;
    float acc[PER];
#pragma unroll
    for (int j = 0; j < PER; ++j) acc[j] = 0.f;
    for (int j0 = 0; j0 < n_all; j0 += 32) {
        const int nb = min(32, n_all - j0);
        if (lane < nb) {
            const int j = j0 + lane;
            int64_t row;
            const float* base;
            const float* lbase;
            if (j < ns * seg_chunks) {
                row = ((int64_t)req_seg_pos[s0 + j / seg_chunks] * q_heads + h) * seg_chunks + j % seg_chunks;
                base = seg_o;
                lbase = seg_lse;
            } else {
                row = (int64_t)bh * n_chunks + (j - ns * seg_chunks);
                base = tail_o;
                lbase = tail_lse;
            }
            sL[lane] = lbase[row];
            sSrc[lane] = base + row * D;
        }
        __syncwarp();
        float mb = m;
        for (int j = 0; j < nb; ++j) mb = fmaxf(mb, sL[j]);
        if (mb != -INFINITY) {
            const float a = m == -INFINITY ? 0.f : rc::fast_exp2(m - mb);
            wsum *= a;
#pragma unroll
            for (int k = 0; k < PER; ++k) acc[k] *= a;
            m = mb;
#pragma unroll 4
            for (int j = 0; j < nb; ++j) {
                const float l2 = sL[j];
                if (l2 == -INFINITY) continue;
                const float w = rc::fast_exp2(l2 - m);
                wsum += w;
                const float* src = sSrc[j] + lane;
#pragma unroll
                for (int k = 0; k < PER; ++k) acc[k] += w * src[32 * k];
            }
        }
        __syncwarp();
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int j = 0; j < PER; ++j) out[(int64_t)bh * D + lane + 32 * j] = __float2bfloat16_rn(acc[j] * inv);
    if (lse && lane == 0) lse[bh] = wsum > 0.f ? (m + log2f(wsum)) * rc::kLn2 : -INFINITY;
}

// ------------------------------------------------------------------ planning
struct DecodePlan {
    int chunk = 0, n_chunks = 0;        // table part: keys per CTA, CTAs per row
    int seg_chunk = 0, seg_chunks = 0;  // cascade: keys per CTA, CTAs per segment
    bool fused = false;                 // one CTA per (row, KV head): no merge pass
    size_t tail_o = 0, tail_lse = 0, seg_o = 0, seg_lse = 0, total = 0;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

rc_status plan_decode(const rc_attn_desc* d, int32_t batch, int32_t max_len, const rc_cascade* casc,
                      DecodePlan* pl) {
    if (!d || batch < 0 || max_len < 0) return RC_ERR_ARG;
    const int hkv = d->pool.kv_heads;
    if (hkv <= 0 || d->q_heads <= 0 || d->q_heads % hkv) return RC_ERR_ARG;
    const int dv = d->pool.head_dim_v;
    const int64_t sms = rc_host::sm_count();
    // Table part: one warp per (row, KV head) when that already gives every
    // SM eight warps (the merge is then fused); otherwise split the keys so
    // that the items just fill one wave of CTAs (a warp's time grows with its
    // tiles, about 2.5 us per 16 keys when the gather saturates HBM, so the
    // wave's longest item sets the call), down to 64 keys per chunk.
    const int64_t base = (int64_t)batch * hkv;
    int64_t splits = 1;
    if (base < 8 * sms) {
        splits = base > 0 ? (kWarpsPerCta * sms) / base : 1;
        const int64_t max_splits = max_len > 0 ? (max_len + kDecKeys - 1) / kDecKeys : 1;
        if (splits > max_splits) splits = max_splits;
        if (splits < 1) splits = 1;
    }
    int64_t chunk = max_len > 0 ? (max_len + splits - 1) / splits : kDecKeys;
    chunk = (chunk + kDecKeys - 1) / kDecKeys * kDecKeys;
    pl->chunk = (int)chunk;
    pl->n_chunks = max_len > 0 ? (int)((max_len + chunk - 1) / chunk) : 1;
    pl->fused = pl->n_chunks == 1;
    // Cascade part: split each segment's keys so that the grid fills the SMs
    // once (one CTA per SM: a second, partial wave would double the time),
    // and in any case so that no CTA takes more than about kSegKeys keys: a
    // CTA's time grows with its tiles, and with many segments (a grid of
    // several waves anyway) a long one would otherwise run all its keys in
    // one CTA while the short ones finish early.  Chunks past a segment's end
    // are empty CTAs that leave at once.
    constexpr int64_t kSegKeys = 512;
    pl->seg_chunk = 0;
    pl->seg_chunks = 1;
    if (casc && casc->n_seg > 0 && casc->max_seg_len > 0) {
        const int G = d->q_heads / hkv;
        const int64_t row_blocks = (casc->max_seg_rows * (int64_t)G + rc_tc2::ROWS - 1) / rc_tc2::ROWS;
        const int64_t cbase = (int64_t)casc->n_seg * row_blocks * hkv;
        int64_t sc = cbase > 0 ? sms / cbase : 1;
        const int64_t sc_len = (casc->max_seg_len + kSegKeys - 1) / kSegKeys;
        if (sc < sc_len) sc = sc_len;
        const int64_t sc_max = (casc->max_seg_len + 255) / 256;
        if (sc > sc_max) sc = sc_max;
        if (sc < 1) sc = 1;
        int64_t len = (casc->max_seg_len + sc - 1) / sc;
        len = (len + rc_tc2::TN - 1) / rc_tc2::TN * rc_tc2::TN;
        pl->seg_chunk = (int)len;
        pl->seg_chunks = (int)((casc->max_seg_len + len - 1) / len);
    }
    const size_t rows = (size_t)batch * d->q_heads;
    pl->tail_o = pl->fused ? 0 : align256(rows * pl->n_chunks * dv * sizeof(float));
    pl->tail_lse = pl->fused ? 0 : align256(rows * pl->n_chunks * sizeof(float));
    const size_t srows = casc && casc->n_seg > 0 ? (size_t)casc->total_seg_rows * d->q_heads * pl->seg_chunks : 0;
    pl->seg_o = align256(srows * dv * sizeof(float));
    pl->seg_lse = align256(srows * sizeof(float));
    pl->total = pl->tail_o + pl->tail_lse + pl->seg_o + pl->seg_lse;
    if (pl->total == 0) pl->total = 256;
    return RC_OK;
}

// after_cascade: launched as the programmatic dependent of the cascade kernel
// just queued on the stream, so that its CTAs start on SMs the cascade leaves
// free and as cascade CTAs finish, instead of after the whole cascade grid.
template <int D, int G, bool FUSED, bool FP8>
cudaError_t launch_split(const DecParams& p, int batch, int kv_heads, cudaStream_t st, bool after_cascade) {
    constexpr int smem = dec_smem_bytes<D, FP8>();
    cudaError_t e = rc_host::ensure_smem<decode_split_kernel<D, G, FUSED, FP8>>(smem);
    if (e != cudaSuccess) return e;
    const int n_items = batch * kv_heads * p.n_chunks;
    const int grid = (n_items + kWarpsPerCta - 1) / kWarpsPerCta;
    if (!after_cascade) {
        decode_split_kernel<D, G, FUSED, FP8><<<grid, 32 * kWarpsPerCta, smem, st>>>(p, n_items);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(32 * kWarpsPerCta);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, decode_split_kernel<D, G, FUSED, FP8>, p, n_items);
}

template <int D, int G, bool FP8>
cudaError_t launch_cascade(const rc::MQParams& p0, const rc_cascade* c, int kv_heads, cudaStream_t st) {
    constexpr int smem = rc_tc2::smem_bytes<D, FP8>();
    cudaError_t e = rc_host::ensure_smem<rc_tc2::attn_tc2_kernel<D, G, rc::MQMode::kCascade, FP8>>(smem);
    if (e != cudaSuccess) return e;
    constexpr int TPC = rc_tc2::ROWS / G;
    rc::MQParams p = p0;
    dim3 grid((c->max_seg_rows + TPC - 1) / TPC, kv_heads, c->n_seg * p.seg_chunks);
    p.n_seg = c->n_seg;
    p.seg_items = 0;
    if (c->host_seg_indptr && c->host_seg_row_indptr) {
        // one CTA per non-empty (segment, key chunk, row block), counted the
        // way the kernel counts them from the device arrays
        int64_t items = 0;
        for (int s = 0; s < c->n_seg; ++s) {
            const int64_t rows = (int64_t)c->host_seg_row_indptr[s + 1] - c->host_seg_row_indptr[s];
            const int64_t len = (int64_t)c->host_seg_indptr[s + 1] - c->host_seg_indptr[s];
            if (rows <= 0) continue;
            int64_t ch = len > 0 ? (len + p.seg_chunk - 1) / p.seg_chunk : 1;
            if (ch > p.seg_chunks) ch = p.seg_chunks;
            items += ch * ((rows + TPC - 1) / TPC);
        }
        if (items > 0 && items <= 0x7fffffff) {
            grid = dim3((unsigned)items, kv_heads, 1);
            p.seg_items = (int32_t)items;
        }
    }
    // programmatic dependent of the previous kernel on the stream (the kernel
    // waits for it before reading anything)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(rc_tc2::THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, rc_tc2::attn_tc2_kernel<D, G, rc::MQMode::kCascade, FP8>, p);
}

template <int D, int G>
cudaError_t run_gqa(const DecParams& dp, const rc::MQParams& mp, const rc_cascade* casc, bool fused, bool fp8,
                    int batch, int kv_heads, cudaStream_t st) {
    cudaError_t e = cudaSuccess;
    const bool with_cascade = casc && casc->n_seg > 0 && casc->max_seg_rows > 0;
    if constexpr (D == 128) {
        if (fp8) {
            if (with_cascade) e = launch_cascade<D, G, true>(mp, casc, kv_heads, st);
            if (e != cudaSuccess) return e;
            return fused ? launch_split<D, G, true, true>(dp, batch, kv_heads, st, with_cascade)
                         : launch_split<D, G, false, true>(dp, batch, kv_heads, st, with_cascade);
        }
    }
    if (with_cascade) e = launch_cascade<D, G, false>(mp, casc, kv_heads, st);
    if (e != cudaSuccess) return e;
    return fused ? launch_split<D, G, true, false>(dp, batch, kv_heads, st, with_cascade)
                 : launch_split<D, G, false, false>(dp, batch, kv_heads, st, with_cascade);
}

template <int D>
cudaError_t dispatch_group(int G, const DecParams& dp, const rc::MQParams& mp, const rc_cascade* casc, bool fused,
                           bool fp8, int batch, int kv_heads, cudaStream_t st, bool* ok) {
    *ok = true;
    switch (G) {
        case 1: return run_gqa<D, 1>(dp, mp, casc, fused, fp8, batch, kv_heads, st);
        case 2: return run_gqa<D, 2>(dp, mp, casc, fused, fp8, batch, kv_heads, st);
        case 4: return run_gqa<D, 4>(dp, mp, casc, fused, fp8, batch, kv_heads, st);
        case 8: return run_gqa<D, 8>(dp, mp, casc, fused, fp8, batch, kv_heads, st);
        default: *ok = false; return cudaSuccess;
    }
}

}  // namespace

extern "C" rc_status attn_decode_workspace(const rc_attn_desc* desc, int32_t batch, int32_t max_len,
                                           const rc_cascade* cascade, size_t* bytes) {
    if (!bytes) return RC_ERR_ARG;
    if (desc && desc->pool.mla) {
        if (batch < 0 || max_len < 0 || desc->q_heads <= 0) return RC_ERR_ARG;
        if (cascade && cascade->n_seg > 0) return RC_ERR_UNSUPPORTED;
        *bytes = rc_host::mla_workspace(batch, desc->q_heads, max_len);
        return RC_OK;
    }
    DecodePlan pl;
    rc_status s = plan_decode(desc, batch, max_len, cascade, &pl);
    if (s != RC_OK) return s;
    *bytes = pl.total;
    return RC_OK;
}

namespace {

// early: the kernel queued just before is the previous step's table pass
// (see MQParams::early)
rc_status decode_impl(const rc_attn_desc* desc, const void* q, const void* k_new, const void* v_new,
                      const rc_kv_table* kv, int32_t batch, const rc_cascade* casc, void* out, float* lse, void* ws,
                      size_t ws_bytes, rc_stream_t stream, bool early = false) {
    if (!desc || !kv || batch < 0) return RC_ERR_ARG;
    if (batch == 0) return RC_OK;
    if (!q || !out || !kv->slots || !kv->start || !kv->len || !desc->pool.k) return RC_ERR_ARG;
    const bool use_casc = casc && casc->n_seg > 0;
    if (desc->pool.mla) {  // one latent KV head: its own kernel (attn_decode_mla.cu)
        if (k_new || desc->pool.kv_fp8) return RC_ERR_UNSUPPORTED;
        if (use_casc) return RC_ERR_UNSUPPORTED;
        if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255)) return RC_ERR_ARG;
        return rc_host::mla_decode(desc, q, kv, batch, out, lse, ws, ws_bytes, (cudaStream_t)stream);
    }
    DecodePlan pl;
    rc_status s = plan_decode(desc, batch, kv->max_len, use_casc ? casc : nullptr, &pl);
    if (s != RC_OK) return s;
    if (!ws || ws_bytes < pl.total) return RC_ERR_ARG;
    if (reinterpret_cast<uintptr_t>(ws) & 255) return RC_ERR_ARG;
    if (use_casc && (!casc->seg_slots || !casc->seg_indptr || !casc->seg_row_indptr || !casc->seg_rows ||
                     !casc->req_seg_indptr || !casc->req_seg_pos))
        return RC_ERR_ARG;
    const rc_pool_desc& P = desc->pool;
    const int D = P.head_dim_k;
    if (P.mla || P.head_dim_v != D || !P.v) return RC_ERR_UNSUPPORTED;
    const bool fp8 = P.kv_fp8 != 0;
    if (fp8) {  // E4M3 pool: the table pass and the cascade read codes and scales
        if (D != 128 || k_new) return RC_ERR_UNSUPPORTED;
        if (!P.k_scale || !P.v_scale) return RC_ERR_ARG;
        if (use_casc && !rc_tc2::fp8_cascade_supported()) return RC_ERR_UNSUPPORTED;
    }
    const int G = desc->q_heads / P.kv_heads;
    unsigned char* w = static_cast<unsigned char*>(ws);
    float* seg_o = reinterpret_cast<float*>(w + pl.tail_o + pl.tail_lse);
    float* seg_lse = reinterpret_cast<float*>(w + pl.tail_o + pl.tail_lse + pl.seg_o);
    DecParams dp;
    dp.q = static_cast<const __nv_bfloat16*>(q);
    dp.pool_k = static_cast<const __nv_bfloat16*>(P.k);
    dp.pool_v = static_cast<const __nv_bfloat16*>(P.v);
    dp.n_slots = P.n_slots;
    dp.kv_heads = P.kv_heads;
    dp.q_heads = desc->q_heads;
    dp.scale_log2 = desc->sm_scale * rc::kLog2e;
    dp.err = P.err;
    dp.table = kv->slots;
    dp.start = kv->start;
    dp.len = kv->len;
    dp.table_len = kv->table_len;
    dp.chunk = pl.chunk;
    dp.n_chunks = pl.n_chunks;
    dp.part_o = reinterpret_cast<float*>(w);
    dp.part_lse = reinterpret_cast<float*>(w + pl.tail_o);
    dp.seg_o = seg_o;
    dp.seg_lse = seg_lse;
    dp.req_seg_indptr = use_casc ? casc->req_seg_indptr : nullptr;
    dp.req_seg_pos = use_casc ? casc->req_seg_pos : nullptr;
    dp.seg_chunks = pl.seg_chunks;
    dp.out = static_cast<__nv_bfloat16*>(out);
    dp.lse = lse;
    dp.k_new = static_cast<const __nv_bfloat16*>(k_new);
    dp.v_new = static_cast<const __nv_bfloat16*>(v_new);
    dp.k_scale = fp8 ? P.k_scale : nullptr;
    dp.v_scale = fp8 ? P.v_scale : nullptr;
    rc::MQParams mp{};
    mp.q = dp.q;
    mp.pool_k = dp.pool_k;
    mp.pool_v = dp.pool_v;
    mp.n_slots = dp.n_slots;
    mp.kv_heads = dp.kv_heads;
    mp.q_heads = dp.q_heads;
    mp.scale_log2 = dp.scale_log2;
    mp.err = dp.err;
    mp.k_scale = dp.k_scale;
    mp.v_scale = dp.v_scale;
    if (use_casc) {
        mp.seg_slots = casc->seg_slots;
        mp.seg_indptr = casc->seg_indptr;
        mp.seg_row_indptr = casc->seg_row_indptr;
        mp.seg_rows = casc->seg_rows;
        mp.part_o = seg_o;
        mp.part_lse = seg_lse;
        mp.seg_chunk = pl.seg_chunk;
        mp.seg_chunks = pl.seg_chunks;
        mp.early = early ? 1 : 0;
    }
    cudaStream_t st = (cudaStream_t)stream;
    bool ok = false;
    cudaError_t e = cudaSuccess;
    const rc_cascade* cc = use_casc ? casc : nullptr;
    if (D == 128) e = dispatch_group<128>(G, dp, mp, cc, pl.fused, fp8, batch, P.kv_heads, st, &ok);
    else if (D == 64) e = dispatch_group<64>(G, dp, mp, cc, pl.fused, false, batch, P.kv_heads, st, &ok);
    if (!ok) return RC_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return RC_ERR_CUDA;
    if (pl.fused) return RC_OK;
    const int32_t* ri = use_casc ? casc->req_seg_indptr : nullptr;
    const int32_t* rp = use_casc ? casc->req_seg_pos : nullptr;
    const unsigned nbh = (unsigned)batch * desc->q_heads;
    __nv_bfloat16* o = static_cast<__nv_bfloat16*>(out);
    // the merge is the split pass's programmatic dependent (it waits for it
    // inside), so its CTAs start as the split pass's leave
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nbh);
    cfg.blockDim = dim3(32);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (D == 128)
        e = cudaLaunchKernelEx(&cfg, merge_kernel<128>, (const float*)dp.part_o, (const float*)dp.part_lse,
                               dp.n_chunks, dp.chunk, dp.len, (const float*)seg_o, (const float*)seg_lse,
                               pl.seg_chunks, ri, rp, desc->q_heads, dp.start, dp.table_len, o, lse, P.err);
    else
        e = cudaLaunchKernelEx(&cfg, merge_kernel<64>, (const float*)dp.part_o, (const float*)dp.part_lse,
                               dp.n_chunks, dp.chunk, dp.len, (const float*)seg_o, (const float*)seg_lse,
                               pl.seg_chunks, ri, rp, desc->q_heads, dp.start, dp.table_len, o, lse, P.err);
    return rc_host::launch_status(e);
}

}  // namespace

extern "C" rc_status attn_decode(const rc_attn_desc* desc, const void* q, const rc_kv_table* kv, int32_t batch,
                                 const rc_cascade* casc, void* out, float* lse, void* ws, size_t ws_bytes,
                                 rc_stream_t stream) {
    return decode_impl(desc, q, nullptr, nullptr, kv, batch, casc, out, lse, ws, ws_bytes, stream);
}

extern "C" rc_status attn_decode_append(const rc_attn_desc* desc, const void* q, const void* k_new,
                                        const void* v_new, const rc_kv_table* kv, int32_t batch,
                                        const rc_cascade* casc, void* out, float* lse, void* ws, size_t ws_bytes,
                                        rc_stream_t stream) {
    if (!k_new || !v_new) return RC_ERR_ARG;
    if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15) return RC_ERR_ARG;
    return decode_impl(desc, q, k_new, v_new, kv, batch, casc, out, lse, ws, ws_bytes, stream);
}

extern "C" rc_status attn_decode_steps(const rc_attn_desc* desc, const rc_kv_table* kv, int32_t batch,
                                       const rc_cascade* casc, const rc_decode_step* steps, int32_t n_steps,
                                       void* ws, size_t ws_bytes, rc_stream_t stream, int32_t* n_done) {
    if (n_done) *n_done = 0;
    if (!desc || !kv || n_steps < 0 || (n_steps > 0 && !steps)) return RC_ERR_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    for (int32_t i = 0; i < n_steps; ++i) {
        const rc_decode_step& s = steps[i];
        if (s.ev_begin && cudaEventRecord((cudaEvent_t)s.ev_begin, st) != cudaSuccess) return RC_ERR_CUDA;
        rc_kv_table t = *kv;
        t.len = s.len;
        t.max_len = s.max_len;
        rc_status r;
        if (s.store_slots) {
            r = kv_store(&desc->pool, s.store_slots, s.k_new, s.v_new, batch, nullptr, nullptr, stream);
            if (r == RC_OK) r = attn_decode(desc, s.q, &t, batch, casc, s.out, s.lse, ws, ws_bytes, stream);
        } else if (s.k_new) {
            if ((reinterpret_cast<uintptr_t>(s.k_new) | reinterpret_cast<uintptr_t>(s.v_new)) & 15 || !s.v_new) {
                r = RC_ERR_ARG;
            } else {
                // after an append step with no event in between, the kernel queued
                // last is that step's table pass (or its merge): this step's
                // cascade may read before waiting for it
                const rc_decode_step* pv = i > 0 ? &steps[i - 1] : nullptr;
                const bool early = pv && pv->k_new && !pv->store_slots && !pv->ev_end && !s.ev_begin;
                r = decode_impl(desc, s.q, s.k_new, s.v_new, &t, batch, casc, s.out, s.lse, ws, ws_bytes, stream,
                                early);
            }
        } else {
            r = attn_decode(desc, s.q, &t, batch, casc, s.out, s.lse, ws, ws_bytes, stream);
        }
        if (r != RC_OK) return r;
        if (s.ev_end && cudaEventRecord((cudaEvent_t)s.ev_end, st) != cudaSuccess) return RC_ERR_CUDA;
        if (n_done) *n_done = i + 1;
    }
    return RC_OK;
}

// ---------------------------------------------------------------------------
// Allocation-free variant.  The split partials go to a file-scope device
// array instead of a caller workspace.  In host code the array's name is only
// a host-side stand-in, so its device address is looked up once per device
// (with that device current) and passed to the kernels like any workspace.

#include <mutex>

namespace {

static __device__ __align__(256) unsigned char rc_decode_scratch[RC_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {nullptr};
std::mutex g_scratch_mu;

rc_status scratch_for_current_device(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return RC_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return RC_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, rc_decode_scratch) != cudaSuccess || !p) return RC_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return RC_OK;
}

}  // namespace

extern "C" rc_status attn_decode_static(const rc_attn_desc* desc, const void* q, const rc_kv_table* kv,
                                        int32_t batch, const rc_cascade* casc, void* out, float* lse,
                                        rc_stream_t stream) {
    if (!desc || !kv || batch < 0) return RC_ERR_ARG;
    if (batch == 0) return RC_OK;
    const rc_cascade* cc = casc && casc->n_seg > 0 ? casc : nullptr;  // as attn_decode plans it
    size_t need = 0;
    rc_status s = attn_decode_workspace(desc, batch, kv->max_len, cc, &need);
    if (s != RC_OK) return s;
    if (need > (size_t)RC_STATIC_SCRATCH_BYTES) return RC_ERR_SCRATCH;
    void* ws = nullptr;
    s = scratch_for_current_device(&ws);
    if (s != RC_OK) return s;
    return attn_decode(desc, q, kv, batch, casc, out, lse, ws, (size_t)RC_STATIC_SCRATCH_BYTES, stream);
}
