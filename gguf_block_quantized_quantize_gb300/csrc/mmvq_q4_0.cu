// MMVQ instantiations for Q4_0 weights (see mmvq.cuh and mmvq_mma_sb.cuh).
#include "mmvq_mma_sb.cuh"

namespace gg {

cudaError_t launch_mmvq_q4_0(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
    // mmvq_tc_min_m..8 tokens on the int8 tensor-core MMVQ (rows of whole
    // 256-value items, 2048 rows or more to fill the GPU)
    if (m >= option_mmvq_tc_min_m() && m <= 8 && sg.rows() >= 2048 && option_mmvq_tc() && mma_sb_fits(GGUF_Q4_0, sg, k, m))
        return launch_mmvq_mma_sb<GGUF_Q4_0>(sg, k, xq, m, yt, s);
    // measured on GB300 (4096 / 14336 rows of 4096 values, 4096 rows of
    // 14336): two rows in flight per register set for 1..2 tokens, four for
    // 3..4 tokens, and 5..8 tokens on one thread per piece
    return launch_mmvq_pt<Q40Piece>(sg, k, xq, m, yt, s, k / 32 * Q4_0_BYTES, MmvqTune{false, false, false, false, false, true});
}

cudaError_t launch_mmvq_routes_q4_0(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s) {
    return launch_mmvq_routes_pt<Q40Piece>(bank, rt, n, k, k / 32 * Q4_0_BYTES, xq, routes, z, s);
}

}  // namespace gg
