// MMVQ instantiations for Q8_0 weights (see mmvq.cuh).
#include "mmvq.cuh"

namespace gg {

cudaError_t launch_mmvq_q8_0(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
    const int64_t n = sg.rows();
    // 5..8 tokens: two threads per piece (4 tokens each) below 4096 rows, one above (measured)
    return launch_mmvq_pt<Q80Piece>(sg, k, xq, m, yt, s, k / 32 * Q8_0_BYTES, MmvqTune{false, false, false, n < 4096});
}

cudaError_t launch_mmvq_routes_q8_0(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s) {
    return launch_mmvq_routes_pt<Q80Piece>(bank, rt, n, k, k / 32 * Q8_0_BYTES, xq, routes, z, s);
}

}  // namespace gg
