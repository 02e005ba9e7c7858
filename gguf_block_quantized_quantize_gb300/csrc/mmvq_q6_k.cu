// MMVQ instantiations for Q6_K weights (see mmvq.cuh).
#include "mmvq.cuh"

namespace gg {

cudaError_t launch_mmvq_q6_k(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
    const int64_t n = sg.rows();
    // 5..8 tokens: two threads per piece below 2048 rows; 2 tokens: four rows per group (measured)
    return launch_mmvq_pt<Q6KPiece>(sg, k, xq, m, yt, s, k / 256 * Q6_K_BYTES, MmvqTune{false, false, n < 2048, n >= 2048, false});
}

}  // namespace gg
