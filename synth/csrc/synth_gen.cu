// GPU and host restatement of the synthetic input definitions in
// synth/hashgen.py (prefix hash, Irwin-Hall bf16 values, next-token model),
// for inputs too large to draw with numpy.  Integer arithmetic throughout, so
// both versions agree bit for bit.  No attention or cache arithmetic here.

#include <cuda_runtime.h>
#include <stdint.h>

namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;
constexpr uint64_t kTokenSalt = 0xD1B54A32D192ED03ull;

__host__ __device__ inline uint64_t mix64(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// One element: token hash h, key = ((layer*4 + kind)*256 + head)*1024 + dim.
__device__ inline uint16_t value_bits(uint64_t h, uint64_t key) {
    int64_t sum = 0;
#pragma unroll
    for (int j = 0; j < 3; ++j) {
        const uint64_t w = mix64(h + (key * 3 + j + 1) * kGamma);
#pragma unroll
        for (int q = 0; q < 4; ++q) sum += (int64_t)((w >> (16 * q)) & 0xFFFF);
    }
    const float v = (float)(sum - 6 * 65536) / 65536.0f;  // exact
    uint32_t b = __float_as_uint(v);
    b = (b + 0x7FFFu + ((b >> 16) & 1u)) >> 16;          // round to nearest even
    return (uint16_t)b;
}

// out[t * out_stride + head * dims + dim] for t < n, head < heads, dim < dims
__global__ void gen_kernel(const uint64_t* __restrict__ hashes, int64_t n, int32_t layer, int32_t kind,
                           int32_t heads, int32_t dims, int32_t head0, uint16_t* __restrict__ out,
                           int64_t out_stride) {
    const int64_t per = (int64_t)heads * dims;
    const int64_t total = n * per;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per;
        const int32_t e = (int32_t)(i - t * per);
        const int32_t head = e / dims, dim = e % dims;
        const uint64_t key = ((uint64_t)(layer * 4 + kind) * 256 + (uint64_t)(head0 + head)) * 1024 + dim;
        out[t * out_stride + e] = value_bits(hashes[t], key);
    }
}

}  // namespace

extern "C" {

// Prefix hashes of tok[0..n) continuing from state h_prev.
void synth_prefix_hashes(const int32_t* tok, int64_t n, uint64_t h_prev, uint64_t* out) {
    uint64_t h = h_prev;
    for (int64_t i = 0; i < n; ++i) {
        h = mix64(h ^ mix64(((uint64_t)(int64_t)tok[i] + 1) * kGamma));
        out[i] = h;
    }
}

// Extend a sequence by `m` tokens of the synthetic model: out_tok[i] is the
// token after the prefix whose hash is the previous state; out_hash[i] the
// hash after appending it.  Starts from state h (the hash of the prompt).
void synth_decode_tokens(uint64_t h, int64_t m, int32_t vocab, int32_t* out_tok, uint64_t* out_hash) {
    for (int64_t i = 0; i < m; ++i) {
        const int32_t y = (int32_t)(mix64(h ^ kTokenSalt) % (uint64_t)vocab);
        out_tok[i] = y;
        h = mix64(h ^ mix64(((uint64_t)(int64_t)y + 1) * kGamma));
        out_hash[i] = h;
    }
}

int synth_gen_values(const uint64_t* d_hashes, int64_t n, int32_t layer, int32_t kind, int32_t heads,
                     int32_t dims, int32_t head0, uint16_t* d_out, int64_t out_stride, void* stream) {
    if (n <= 0) return 0;
    const int64_t total = n * heads * dims;
    int64_t blocks = (total + 255) / 256;
    if (blocks > 65536) blocks = 65536;
    gen_kernel<<<(unsigned)blocks, 256, 0, (cudaStream_t)stream>>>(d_hashes, n, layer, kind, heads, dims, head0,
                                                                  d_out, out_stride);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // extern "C"
