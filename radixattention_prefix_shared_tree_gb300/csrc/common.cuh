// Device helpers shared by the kernels of the library (sm_103a).
#pragma once

#include <cuda_runtime.h>
#include <utility>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "../../include/radixattn.h"

#define RC_DEV __device__ __forceinline__

namespace rc {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Error bits OR-ed into the caller's device error word.
constexpr int32_t kErrBadSlot = 1;
constexpr int32_t kErrTimeout = 2;

RC_DEV void flag_error(int32_t* err, int32_t bit) {
    if (err) atomicOr(err, bit);
}

RC_DEV uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte asynchronous copy global -> shared; src_bytes = 0 writes zeros.
RC_DEV void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes)
                 : "memory");
}
// The same with constant byte offsets added to both addresses inside the
// instruction ([reg+imm] addressing): a fully unrolled run of copies then
// costs one instruction each.
template <int DST_OFF, int SRC_OFF>
RC_DEV void cp_async16_at(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0+%3], [%1+%4], 16, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes),
                 "n"(DST_OFF), "n"(SRC_OFF)
                 : "memory");
}
// N copies i = 0..N-1 at dst + i * DST_STEP and src + i * SRC_STEP bytes.
template <int DST_STEP, int SRC_STEP, int... I>
RC_DEV void cp_async16_run(uint32_t dst, const void* src, uint32_t src_bytes, std::integer_sequence<int, I...>) {
    (cp_async16_at<I * DST_STEP, I * SRC_STEP>(dst, src, src_bytes), ...);
}
// The same with an L2 eviction-priority policy (from l2_policy_*).
RC_DEV void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0], [%1], 16, %2, %3;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes), "l"(policy)
                 : "memory");
}
// cp_async16_at / cp_async16_run with an L2 eviction-priority policy.
template <int DST_OFF, int SRC_OFF>
RC_DEV void cp_async16_at(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t policy) {
    asm volatile("cp.async.cg.shared.global.L2::cache_hint [%0+%4], [%1+%5], 16, %2, %3;\n" ::"r"(dst), "l"(src),
                 "r"(src_bytes), "l"(policy), "n"(DST_OFF), "n"(SRC_OFF)
                 : "memory");
}
template <int DST_STEP, int SRC_STEP, int... I>
RC_DEV void cp_async16_run(uint32_t dst, const void* src, uint32_t src_bytes, uint64_t policy,
                           std::integer_sequence<int, I...>) {
    (cp_async16_at<I * DST_STEP, I * SRC_STEP>(dst, src, src_bytes, policy), ...);
}
// L2 policies: lines a kernel reads once (a request's private keys, which
// stream through) go first; lines many CTAs and the next step read again
// (a shared prefix) stay.
RC_DEV uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}
RC_DEV uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}
// Bring `bytes` (a multiple of 16) at a 16-byte aligned global address into
// L2 ahead of the copies that will read them; nothing lands in shared memory.
RC_DEV void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;\n" ::"l"(src), "r"(bytes) : "memory");
}
// 4-byte asynchronous copy (slot ids); src_bytes = 0 writes zero.
RC_DEV void cp_async4(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
RC_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
RC_DEV void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

RC_DEV void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
RC_DEV void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
RC_DEV void ldmatrix_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];\n"
                 : "=r"(r0), "=r"(r1)
                 : "r"(addr));
}

// Transpose of an 8x8 b16 matrix held as one register per thread in the
// ldmatrix fragment layout.
RC_DEV uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// D = A(16x16 bf16, row) * B(16x8 bf16, col) + D, fp32 accumulate.
RC_DEV void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                           uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same with f16 operands.
RC_DEV void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                          uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

RC_DEV uint32_t pack_f16(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Two E4M3 codes (low byte first) to two f16 (low half first); exact, since
// every E4M3 value is an f16 value.
RC_DEV uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    uint32_t d;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, lo;\n\t}\n"
        : "=r"(d)
        : "r"(two_codes));
    return d;
}
// Four E4M3 codes (one word, low byte first) to two f16 pairs: lo gets codes
// 0 and 1, hi codes 2 and 3.
RC_DEV void e4m3x4_to_f16x4(uint32_t four_codes, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.rn.f16x2.e4m3x2 %0, a;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, b;\n\t}\n"
        : "=r"(lo), "=r"(hi)
        : "r"(four_codes));
}

// A bf16 pair to an f16 pair (exact while |x| is within f16's range).
RC_DEV uint32_t bf16x2_to_f16x2(uint32_t w) {
    return pack_f16(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// Byte permute: byte i of the result is byte sel.nibble[i] of {b:a}.
RC_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

RC_DEV uint32_t pack_bf16(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

RC_DEV float fast_exp2(float x) { return exp2f(x); }

// Byte offset of 16-byte chunk `c` of row `r` in a tile whose rows are
// `chunks` 16-byte chunks long, XOR-swizzled on the low three bits so that
// ldmatrix over 8 consecutive rows touches 8 different bank groups.
template <int CHUNKS>
RC_DEV uint32_t swz(int r, int c) {
    return static_cast<uint32_t>((r * CHUNKS + (c ^ (r & 7))) * 16);
}

}  // namespace rc

// Host-side launch helpers.
namespace rc_host {
int sm_count();
// latent (MLA) decode, attn_decode_mla.cu
size_t mla_workspace(int32_t batch, int32_t q_heads, int32_t max_len);
rc_status mla_decode(const rc_attn_desc* desc, const void* q, const rc_kv_table* kv, int32_t batch, void* out,
                     float* lse, void* ws, size_t ws_bytes, cudaStream_t st);
inline rc_status launch_status(cudaError_t e) { return e == cudaSuccess ? RC_OK : RC_ERR_CUDA; }

// Raise a kernel's dynamic shared-memory limit once per device (one flag
// array per kernel: the kernel is a template argument).
template <auto Kernel>
cudaError_t ensure_smem(int bytes) {
    static bool done[64] = {false};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}
}  // namespace rc_host
