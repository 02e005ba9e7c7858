// MMVQ instantiations for Q6_K weights (see mmvq.cuh).
#include "mmvq_mma_q6k.cuh"

namespace gg {

constexpr int64_t Q6K_TC_MIN_ROWS = 32768;

cudaError_t launch_mmvq_q6_k(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
    const int64_t n = sg.rows();
    // mmvq_tc_min_m..8 tokens of tall matrices (LM heads): the tensor-core
    // kernel; below 32768 rows the dp4a kernel is as fast or faster (measured)
    if (m >= option_mmvq_tc_min_m() && m <= 8 && n >= Q6K_TC_MIN_ROWS && option_mmvq_tc() && mma_q6k_fits(k, m))
        return launch_mmvq_mma_q6k(sg, k, xq, m, yt, s);
    // 5..8 tokens: two threads per piece below 2048 rows; 2 tokens: four rows per group (measured)
    return launch_mmvq_pt<Q6KPiece>(sg, k, xq, m, yt, s, k / 256 * Q6_K_BYTES, MmvqTune{false, false, false, n < 2048, n >= 2048, false});
}

cudaError_t launch_mmvq_routes_q6_k(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s) {
    return launch_mmvq_routes_pt<Q6KPiece>(bank, rt, n, k, k / 256 * Q6_K_BYTES, xq, routes, z, s);
}

}  // namespace gg
