// MMVQ instantiations for Q4_K weights (see mmvq.cuh and mmvq_mma.cuh).
#include "mmvq_mma.cuh"

namespace gg {

cudaError_t launch_mmvq_q4_k(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
    const int64_t n = sg.rows();
    // 5..8 tokens: exact block dots on the int8 tensor cores when the q8_1 rows
    // fit in shared memory and there are enough 16-row tiles to fill the GPU
    // (below 2048 rows the per-CTA staging of the activations outweighs it)
    if (m >= 5 && n >= 2048 && option_mmvq_tc() && mma_q4k_fits(k))
        return launch_mmvq_mma_q4k(sg, k, xq, m, yt, s);
    return launch_mmvq_pt<Q4KPiece>(sg, k, xq, m, yt, s, k / 256 * Q4_K_BYTES,
                                    MmvqTune{n >= 8192, false, true});
}

}  // namespace gg
