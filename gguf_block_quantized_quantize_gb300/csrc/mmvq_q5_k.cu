// MMVQ instantiations for Q5_K weights (see mmvq.cuh).
#include "mmvq.cuh"

namespace gg {

cudaError_t launch_mmvq_q5_k(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
    // 80 bytes of weights per piece and row: two rows in flight per register
    // set at every token count; 5..8 tokens as two threads per piece
    return launch_mmvq_pt<Q5KPiece>(sg, k, xq, m, yt, s, k / 256 * Q5_K_BYTES, MmvqTune{false, false, true, false, false});
}

cudaError_t launch_mmvq_routes_q5_k(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s) {
    return launch_mmvq_routes_pt<Q5KPiece>(bank, rt, n, k, k / 256 * Q5_K_BYTES, xq, routes, z, s);
}

}  // namespace gg
