// attn_extend: prefill of the new (uncached) tokens of each request over its
// cached prefix.  In inference-notes note 49, section 2, request 2 reuses the
// shared system prompt and "only Q2" has to be computed; in the SageMaker LMI
// article's prefill phase all of those tokens are processed at once.  Token i
// of request b sits at position len[b] - n_b + i of its slot-table row and
// attends causally to positions 0..itself, prefix included.
//
// The kernel body is attn_tc2.cuh: a CTA owns 256 query rows = (256/G new
// tokens) x (the G query heads of one KV head) in two M=128 tiles, so each
// gathered K/V row serves every head of its group and both tiles; both
// products run on tcgen05 with the accumulators in TMEM, with producer,
// MMA and softmax warps; bf16 output written directly (no split, no
// workspace).

#include "attn_tc2.cuh"
#include "common.cuh"

namespace {

template <int D, int G, bool FP8>
cudaError_t launch_extend(const rc::MQParams& p, int batch, int max_q, int kv_heads, cudaStream_t st) {
    constexpr int smem = rc_tc2::smem_bytes<D, FP8>();
    cudaError_t e = rc_host::ensure_smem<rc_tc2::attn_tc2_kernel<D, G, rc::MQMode::kExtend, FP8>>(smem);
    if (e != cudaSuccess) return e;
    constexpr int TPC = rc_tc2::ROWS / G;
    dim3 grid((max_q + TPC - 1) / TPC, kv_heads, batch);
    rc_tc2::attn_tc2_kernel<D, G, rc::MQMode::kExtend, FP8><<<grid, rc_tc2::THREADS, smem, st>>>(p);
    return cudaGetLastError();
}

template <int D, int G>
cudaError_t launch_extend_any(const rc::MQParams& p, bool fp8, int batch, int max_q, int kv_heads, cudaStream_t st) {
    if constexpr (D == 128) {
        if (fp8) return launch_extend<D, G, true>(p, batch, max_q, kv_heads, st);
    }
    return launch_extend<D, G, false>(p, batch, max_q, kv_heads, st);
}

template <int D>
cudaError_t dispatch(int G, const rc::MQParams& p, bool fp8, int batch, int max_q, int kv_heads, cudaStream_t st,
                     bool* ok) {
    *ok = true;
    switch (G) {
        case 1: return launch_extend_any<D, 1>(p, fp8, batch, max_q, kv_heads, st);
        case 2: return launch_extend_any<D, 2>(p, fp8, batch, max_q, kv_heads, st);
        case 4: return launch_extend_any<D, 4>(p, fp8, batch, max_q, kv_heads, st);
        case 8: return launch_extend_any<D, 8>(p, fp8, batch, max_q, kv_heads, st);
        default: *ok = false; return cudaSuccess;
    }
}

}  // namespace

extern "C" rc_status attn_extend_workspace(const rc_attn_desc* desc, int32_t batch, int32_t max_q,
                                           int32_t max_len, size_t* bytes) {
    if (!desc || !bytes || batch < 0 || max_q < 0 || max_len < 0) return RC_ERR_ARG;
    *bytes = 0;
    return RC_OK;
}

extern "C" rc_status attn_extend(const rc_attn_desc* desc, const void* q, const int32_t* qo_indptr,
                                 const rc_kv_table* kv, int32_t batch, int32_t max_q, void* out, float* lse,
                                 void* ws, size_t ws_bytes, rc_stream_t stream) {
    (void)ws;
    (void)ws_bytes;
    if (!desc || !kv || batch < 0 || max_q < 0) return RC_ERR_ARG;
    if (batch == 0 || max_q == 0) return RC_OK;
    if (!q || !qo_indptr || !out || !kv->slots || !kv->start || !kv->len || !desc->pool.k) return RC_ERR_ARG;
    const rc_pool_desc& P = desc->pool;
    if (P.kv_heads <= 0 || desc->q_heads <= 0 || desc->q_heads % P.kv_heads) return RC_ERR_ARG;
    if (P.mla || !P.v || P.head_dim_v != P.head_dim_k) return RC_ERR_UNSUPPORTED;
    const bool fp8 = P.kv_fp8 != 0;
    if (fp8 && P.head_dim_k != 128) return RC_ERR_UNSUPPORTED;
    if (fp8 && (!P.k_scale || !P.v_scale)) return RC_ERR_ARG;
    rc::MQParams p{};
    p.q = static_cast<const __nv_bfloat16*>(q);
    p.pool_k = static_cast<const __nv_bfloat16*>(P.k);
    p.pool_v = static_cast<const __nv_bfloat16*>(P.v);
    p.n_slots = P.n_slots;
    p.kv_heads = P.kv_heads;
    p.q_heads = desc->q_heads;
    p.scale_log2 = desc->sm_scale * rc::kLog2e;
    p.err = P.err;
    p.qo_indptr = qo_indptr;
    p.table = kv->slots;
    p.start = kv->start;
    p.len = kv->len;
    p.table_len = kv->table_len;
    p.out = static_cast<__nv_bfloat16*>(out);
    p.lse = lse;
    p.k_scale = fp8 ? P.k_scale : nullptr;
    p.v_scale = fp8 ? P.v_scale : nullptr;
    const int G = desc->q_heads / P.kv_heads;
    bool ok = false;
    cudaError_t e = cudaSuccess;
    cudaStream_t st = (cudaStream_t)stream;
    if (P.head_dim_k == 128) e = dispatch<128>(G, p, fp8, batch, max_q, P.kv_heads, st, &ok);
    else if (P.head_dim_k == 64) e = dispatch<64>(G, p, false, batch, max_q, P.kv_heads, st, &ok);
    if (!ok) return RC_ERR_UNSUPPORTED;
    return rc_host::launch_status(e);
}
