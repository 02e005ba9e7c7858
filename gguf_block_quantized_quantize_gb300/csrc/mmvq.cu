// MMVQ dispatch by weight type (kernels in mmvq.cuh, one translation unit per type).
#include "mmvq.cuh"

namespace gg {

// One piece per thread and at most 512 threads per CTA: K <= 16384 (longer
// rows take the tensor-core path, which has no K limit).
constexpr int64_t MMVQ_MAX_PIECES = 512;

cudaError_t launch_mmvq(const uint8_t *w, int wt, int64_t n, int64_t k, const uint8_t *xq, int64_t m, void *y,
                        int yt, int64_t ldy, cudaStream_t s) {
    if (n == 0 || m == 0) return cudaSuccess;
    if (k / 32 > MMVQ_MAX_PIECES || m > 8) return cudaErrorInvalidValue;
    switch (wt) {
    case GGUF_Q8_0: return launch_mmvq_q8_0(w, n, k, xq, m, y, yt, ldy, s);
    case GGUF_Q4_K: return launch_mmvq_q4_k(w, n, k, xq, m, y, yt, ldy, s);
    case GGUF_Q6_K: return launch_mmvq_q6_k(w, n, k, xq, m, y, yt, ldy, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gg
