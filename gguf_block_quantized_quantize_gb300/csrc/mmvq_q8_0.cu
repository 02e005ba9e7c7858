// MMVQ instantiations for Q8_0 weights (see mmvq.cuh and mmvq_mma_sb.cuh).
#include "mmvq_mma_sb.cuh"

namespace gg {

cudaError_t launch_mmvq_q8_0(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
    // mmvq_tc_min_m..8 tokens on the int8 tensor-core MMVQ (rows of whole
    // 256-value items, 2048 rows or more to fill the GPU)
    if (m >= option_mmvq_tc_min_m() && m <= 8 && sg.rows() >= 2048 && option_mmvq_tc() && mma_sb_fits(GGUF_Q8_0, sg, k, m))
        return launch_mmvq_mma_sb<GGUF_Q8_0>(sg, k, xq, m, yt, s);
    const int64_t n = sg.rows();
    // 5..8 tokens: two threads per piece (4 tokens each) below 4096 rows, one above (measured)
    return launch_mmvq_pt<Q80Piece>(sg, k, xq, m, yt, s, k / 32 * Q8_0_BYTES, MmvqTune{false, false, false, n < 4096});
}

cudaError_t launch_mmvq_routes_q8_0(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s) {
    return launch_mmvq_routes_pt<Q80Piece>(bank, rt, n, k, k / 32 * Q8_0_BYTES, xq, routes, z, s);
}

}  // namespace gg
