// Oracle for prefix-shared attention: test infrastructure only.
//
// Only the test suite, the package smoke check and the benchmark's CPU-baseline
// leg may load this code; it shares nothing with the product library.
//
// What it computes is the plain definition of attention for one query row
// over the keys it may see (the request's own context: the cached prefix plus,
// for a prefill of new tokens, the new tokens up to and including itself):
//
//     s_j = scale * <q_h, k_{j, g(h)}>,     o_h = sum_j softmax(s)_j v_{j, g(h)}
//
// with g(h) = floor(h * Hkv / Hq) the key/value head that query head h reads
// (grouped-query attention; Hkv = 1 with a 576-wide latent row whose first 512
// columns serve as V is the multi-head-latent case), and lse_h = log sum_j
// exp(s_j).  Prefill and decode differ only in which keys a query sees: the
// pages (SGLang "RadixAttention"; the SageMaker LMI article's prefill/decode
// section) have prefill process all prompt tokens at once and decode one
// token at a time over the cached K/V, and the inference-notes note 49,
// section 2, has only the new part of a request computed while the shared
// part's K/V is reused.
//
// Inputs are bf16 bit patterns, widened exactly; all arithmetic is in double,
// softmax in two passes (max, then sum).  Nothing is blocked or reordered.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

double widen(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    std::memcpy(&f, &u, 4);
    return (double)f;
}

// One query head over ctx keys.  k rows: k + j*k_tok_stride + head*k_head_stride.
void one_head(const uint16_t* q, const uint16_t* k, const uint16_t* v, int64_t ctx,
              int64_t k_tok_stride, int64_t v_tok_stride, int dk, int dv, double scale,
              double* out, double* lse) {
    std::vector<double> s((size_t)ctx);
    double m = -INFINITY;
    for (int64_t j = 0; j < ctx; ++j) {
        double dot = 0.0;
        for (int c = 0; c < dk; ++c) dot += widen(q[c]) * widen(k[j * k_tok_stride + c]);
        s[(size_t)j] = scale * dot;
        if (s[(size_t)j] > m) m = s[(size_t)j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < ctx; ++j) l += std::exp(s[(size_t)j] - m);
    for (int c = 0; c < dv; ++c) out[c] = 0.0;
    for (int64_t j = 0; j < ctx; ++j) {
        double p = std::exp(s[(size_t)j] - m) / l;
        for (int c = 0; c < dv; ++c) out[c] += p * widen(v[j * v_tok_stride + c]);
    }
    if (lse) *lse = m + std::log(l);
}

}  // namespace

extern "C" {

int oracle_num_threads() {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

// Threads of later oracle_attention calls from this thread (n <= 0: all the
// host's cores again); lets the caller time the oracle on one core too.
void oracle_set_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : omp_get_num_procs());
#else
    (void)n;
#endif
}

// Many query rows at once.  Query row r (q + r*Hq*dk) sees keys
// kv_off[r] .. kv_off[r] + ctx[r] - 1 of the token-major arrays
// k [tokens][Hkv][dk] and v [tokens][Hkv][dv] (v may alias k with
// v_tok_stride = Hkv*dk for the latent case).  out: [rows][Hq][dv],
// lse: [rows][Hq] (may be null).  Rows x heads run in parallel with OpenMP;
// each (row, head) pair is computed exactly as above.
void oracle_attention(int64_t rows, const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      const int64_t* kv_off, const int64_t* ctx, int Hq, int Hkv, int dk, int dv,
                      int64_t k_tok_stride, int64_t v_tok_stride, double scale, double* out,
                      double* lse) {
    const int64_t pairs = rows * (int64_t)Hq;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t p = 0; p < pairs; ++p) {
        int64_t r = p / Hq;
        int h = (int)(p % Hq);
        int g = (int)((int64_t)h * Hkv / Hq);
        const uint16_t* qh = q + (r * Hq + h) * (int64_t)dk;
        const uint16_t* kh = k + kv_off[r] * k_tok_stride + (int64_t)g * dk;
        const uint16_t* vh = v + kv_off[r] * v_tok_stride + (int64_t)g * (v == k ? dk : dv);
        one_head(qh, kh, vh, ctx[r], k_tok_stride, v_tok_stride, dk, dv, scale,
                 out + (r * Hq + h) * (int64_t)dv, lse ? lse + r * Hq + h : nullptr);
    }
}

}  // extern "C"
