// MMVQ instantiations for MXFP4 weights (see mmvq.cuh and mmvq_mma_sb.cuh).
#include "mmvq_mma_sb.cuh"

namespace gg {

cudaError_t launch_mmvq_mxfp4(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
    // mmvq_tc_min_m..8 tokens on the int8 tensor-core MMVQ (rows of whole
    // 512-value items, 2048 rows or more to fill the GPU)
    if (m >= option_mmvq_tc_min_m() && m <= 8 && sg.rows() >= 2048 && option_mmvq_tc() &&
        mma_sb_fits(GGUF_MXFP4, sg, k, m))
        return launch_mmvq_mma_sb<GGUF_MXFP4>(sg, k, xq, m, yt, s);
    // Q4_0's configuration (the same two-block staged pieces)
    return launch_mmvq_pt<MX4Piece>(sg, k, xq, m, yt, s, k / 32 * MXFP4_BYTES, MmvqTune{false, false, false, false, false, true});
}

cudaError_t launch_mmvq_routes_mxfp4(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k,
                                     const uint8_t *xq, int64_t routes, float *z, cudaStream_t s) {
    return launch_mmvq_routes_pt<MX4Piece>(bank, rt, n, k, k / 32 * MXFP4_BYTES, xq, routes, z, s);
}

}  // namespace gg
