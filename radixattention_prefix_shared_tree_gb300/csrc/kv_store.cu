// kv_store: scatter the K/V rows of newly computed tokens into their pool
// slots.  In "RadixAttention, eviction and cache churn" (inference-notes note
// 49), section 2, each edge of the radix tree keeps the KV of its tokens; here
// a token's KV is one row per pool array, and the tree (host) only holds the
// slot id.  Pure data movement: every byte is read once and written once, so
// the kernel is bound by HBM bandwidth.  One thread moves one 16-byte chunk;
// consecutive threads move consecutive chunks of a row, so both the read of
// the dense input and the write into the slot's row are fully coalesced.

#include "common.cuh"

namespace {

__global__ void __launch_bounds__(256) kv_store_kernel(const int32_t* __restrict__ slots,
                                                       const uint4* __restrict__ k_new,
                                                       const uint4* __restrict__ v_new,
                                                       uint4* __restrict__ pool_k, uint4* __restrict__ pool_v,
                                                       int64_t n_slots, int32_t n, int32_t k_chunks,
                                                       int32_t v_chunks, int32_t* __restrict__ table,
                                                       const int32_t* __restrict__ table_pos, int32_t* err) {
    const int64_t row_chunks = (int64_t)k_chunks + v_chunks;
    const int64_t total = (int64_t)n * row_chunks;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int32_t t = (int32_t)(i / row_chunks);
        const int32_t c = (int32_t)(i - (int64_t)t * row_chunks);
        const int32_t s = __ldg(slots + t);
        if (s < 0 || (int64_t)s >= n_slots) {
            if (c == 0) rc::flag_error(err, rc::kErrBadSlot);
            continue;
        }
        if (c < k_chunks) {
            pool_k[(int64_t)s * k_chunks + c] = __ldg(k_new + (int64_t)t * k_chunks + c);
        } else {
            const int32_t cv = c - k_chunks;
            pool_v[(int64_t)s * v_chunks + cv] = __ldg(v_new + (int64_t)t * v_chunks + cv);
        }
        if (c == 0 && table) table[__ldg(table_pos + t)] = s;
    }
}

// FP8 pool: one warp per (token, K or V, head) row of 128 values; each lane
// holds four.  scale = amax / 448 and code_i = e4m3(x_i / scale), both
// quotients correctly rounded fp32 divisions, the E4M3 rounding to nearest
// (ties to even) with saturation at +-448; an all-zero row stores scale 0.
__global__ void __launch_bounds__(256) kv_store_fp8_kernel(const int32_t* __restrict__ slots,
                                                           const __nv_bfloat16* __restrict__ k_new,
                                                           const __nv_bfloat16* __restrict__ v_new,
                                                           uint8_t* __restrict__ pool_k, uint8_t* __restrict__ pool_v,
                                                           float* __restrict__ k_scale, float* __restrict__ v_scale,
                                                           int64_t n_slots, int32_t n, int32_t heads,
                                                           int32_t* __restrict__ table,
                                                           const int32_t* __restrict__ table_pos, int32_t* err) {
    constexpr int D = 128;
    const int lane = threadIdx.x & 31;
    const int64_t rows = (int64_t)n * 2 * heads;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows;
         r += ((int64_t)gridDim.x * blockDim.x) >> 5) {
        const int32_t t = (int32_t)(r / (2 * heads));
        const int32_t j = (int32_t)(r - (int64_t)t * 2 * heads);
        const bool is_v = j >= heads;
        const int32_t h = is_v ? j - heads : j;
        const int32_t s = __ldg(slots + t);
        if (s < 0 || (int64_t)s >= n_slots) {
            if (lane == 0 && j == 0) rc::flag_error(err, rc::kErrBadSlot);
            continue;
        }
        const uint2 raw = __ldg(reinterpret_cast<const uint2*>((is_v ? v_new : k_new) +
                                                              ((int64_t)t * heads + h) * D) + lane);
        float x[4] = {__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xffff0000u),
                      __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xffff0000u)};
        float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
        for (int k = 16; k > 0; k >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, k));
        const float scale = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
        uint32_t codes = 0;
        if (scale > 0.f) {
            const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(
                make_float2(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale)), __NV_SATFINITE, __NV_E4M3);
            const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(
                make_float2(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale)), __NV_SATFINITE, __NV_E4M3);
            codes = (uint32_t)lo | ((uint32_t)hi << 16);
        }
        const int64_t row = (int64_t)s * heads + h;
        reinterpret_cast<uint32_t*>((is_v ? pool_v : pool_k) + row * D)[lane] = codes;
        if (lane == 0) (is_v ? v_scale : k_scale)[row] = scale;
        if (lane == 0 && j == 0 && table) table[__ldg(table_pos + t)] = s;
    }
}

}  // namespace

extern "C" rc_status kv_store(const rc_pool_desc* pool, const int32_t* slots, const void* k_new,
                              const void* v_new, int32_t n, int32_t* table, const int32_t* table_pos,
                              rc_stream_t stream) {
    if (!pool || n < 0 || !pool->k || pool->kv_heads <= 0 || pool->head_dim_k <= 0) return RC_ERR_ARG;
    if (n == 0) return RC_OK;
    if (!slots || !k_new) return RC_ERR_ARG;
    if ((table == nullptr) != (table_pos == nullptr)) return RC_ERR_ARG;
    if (pool->kv_fp8) {
        if (pool->mla || pool->head_dim_k != 128 || pool->head_dim_v != 128) return RC_ERR_UNSUPPORTED;
        if (!pool->v || !v_new || !pool->k_scale || !pool->v_scale) return RC_ERR_ARG;
        if ((reinterpret_cast<uintptr_t>(pool->k) | reinterpret_cast<uintptr_t>(pool->v) |
             reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
            return RC_ERR_ARG;
        const int64_t rows = (int64_t)n * 2 * pool->kv_heads;
        const int64_t want = (rows + 7) / 8;
        const int64_t cap = (int64_t)rc_host::sm_count() * 8;
        const int grid = (int)(want < cap ? want : cap);
        kv_store_fp8_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(
            slots, (const __nv_bfloat16*)k_new, (const __nv_bfloat16*)v_new, (uint8_t*)pool->k, (uint8_t*)pool->v,
            pool->k_scale, pool->v_scale, pool->n_slots, n, pool->kv_heads, table, table_pos, pool->err);
        return rc_host::launch_status(cudaGetLastError());
    }
    const int64_t k_bytes = (int64_t)pool->kv_heads * pool->head_dim_k * 2;
    int64_t v_bytes = 0;
    if (!pool->mla) {
        if (!pool->v || !v_new || pool->head_dim_v <= 0) return RC_ERR_ARG;
        v_bytes = (int64_t)pool->kv_heads * pool->head_dim_v * 2;
    }
    if (k_bytes % 16 || v_bytes % 16) return RC_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(pool->k) | reinterpret_cast<uintptr_t>(pool->v) |
         reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new)) & 15)
        return RC_ERR_ARG;
    const int32_t kc = (int32_t)(k_bytes / 16), vc = (int32_t)(v_bytes / 16);
    const int64_t total = (int64_t)n * (kc + vc);
    const int64_t want = (total + 255) / 256;
    const int64_t cap = (int64_t)rc_host::sm_count() * 8;
    const int grid = (int)(want < cap ? want : cap);
    kv_store_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(
        slots, (const uint4*)k_new, (const uint4*)v_new, (uint4*)pool->k, (uint4*)pool->v, pool->n_slots, n, kc,
        vc, table, table_pos, pool->err);
    return rc_host::launch_status(cudaGetLastError());
}
