// MMVQ instantiations for Q5_K weights (see mmvq.cuh and mmvq_mma.cuh).
#include "mmvq_mma.cuh"

namespace gg {

cudaError_t launch_mmvq_q5_k(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
    // mmvq_tc_min_m..8 tokens on the int8 tensor-core MMVQ, as for Q4_K (the
    // q8_1 rows fit in shared memory, and 2048 rows or more fill the GPU)
    if (m >= option_mmvq_tc_min_m() && m <= 8 && sg.rows() >= 2048 && option_mmvq_tc() && mma_q4k_fits(k, m))
        return launch_mmvq_mma_kq<GGUF_Q5_K>(sg, k, xq, m, yt, s);
    // measured on GB300 (4096 and 14336 rows of 4096 values): two rows in
    // flight per register set for 1 and 3..4 tokens, four for 2 tokens
    // (14336 rows: 11.2 -> 10.3 us), and 5..8 tokens on one thread per piece
    // (29.2 -> 24.7 us; two threads with 4 tokens each are slower here)
    return launch_mmvq_pt<Q5KPiece>(sg, k, xq, m, yt, s, k / 256 * Q5_K_BYTES, MmvqTune{false, false, false, false, true, false});
}

cudaError_t launch_mmvq_routes_q5_k(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s) {
    return launch_mmvq_routes_pt<Q5KPiece>(bank, rt, n, k, k / 256 * Q5_K_BYTES, xq, routes, z, s);
}

}  // namespace gg
