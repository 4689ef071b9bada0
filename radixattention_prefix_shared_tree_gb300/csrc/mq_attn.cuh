// Parameters of the many-query-rows attention kernel (attn_tc2.cuh): the
// kernel body of attn_extend (new tokens over their cached prefix, causal
// among themselves) and of the cascade step of attn_decode (a shared prefix
// segment read once for every request that branches below it).
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
    int32_t n_seg;
    // > 0: the grid's x is this many non-empty (segment, key chunk, row block)
    // items, in segment order (within a segment: chunk-major), and z is 1
    int32_t seg_items;
    // cascade, nonzero: the preceding grid on the stream is the previous
    // decode step's table pass, which writes only rows' private keys and reads
    // the partials: the kernel reads Q and the segments before waiting for
    // it, and waits only before its first global write
    int32_t early;
    // FP8 pool: pool_k / pool_v hold E4M3 codes and these the per-row scales
    const float* k_scale;  // [n_slots][kv_heads]
    const float* v_scale;
};

}  // namespace rc
