// MMVQ instantiations for Q4_K weights (see mmvq.cuh).
#include "mmvq.cuh"

namespace gg {

cudaError_t launch_mmvq_q4_k(const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, void *y, int yt,
                             int64_t ldy, cudaStream_t s) {
    return launch_mmvq_pt<Q4KPiece>(w, n, k, xq, m, y, yt, ldy, s, k / 256 * Q4_K_BYTES, MmvqTune{n >= 8192, false, true});
}

}  // namespace gg
