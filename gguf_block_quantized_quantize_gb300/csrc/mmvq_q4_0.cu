// MMVQ instantiations for Q4_0 weights (see mmvq.cuh).
#include "mmvq.cuh"

namespace gg {

cudaError_t launch_mmvq_q4_0(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
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
