// MMVQ instantiations for Q4_K weights (see mmvq.cuh and mmvq_mma.cuh).
#include "mmvq_mma.cuh"

namespace gg {

cudaError_t launch_mmvq_q4_k(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
    const int64_t n = sg.rows();
    // 9..32 tokens: the tensor-core kernel with 2 or 4 n-tiles (the caller
    // checked mmvq_tc_wide); mmvq_tc_min_m..8 tokens: the tensor-core kernel
    // when the q8_1 rows fit in shared memory and there are enough 16-row
    // tiles to fill the GPU (below 2048 rows the per-CTA staging of the
    // activations outweighs it)
    if (m > 8) return mma_q4k_fits(k, m) ? launch_mmvq_mma_kq<GGUF_Q4_K>(sg, k, xq, m, yt, s) : cudaErrorInvalidValue;
    if (m >= option_mmvq_tc_min_m() && n >= 2048 && option_mmvq_tc() && mma_q4k_fits(k, m))
        return launch_mmvq_mma_kq<GGUF_Q4_K>(sg, k, xq, m, yt, s);
    // one token: 8 rows in flight per thread on matrices of 8192 rows or more
    // (GB300, 18432 rows of 4096: 9.5 us against 11.0 with 4 rows)
    return launch_mmvq_pt<Q4KPiece>(sg, k, xq, m, yt, s, k / 256 * Q4_K_BYTES,
                                    MmvqTune{n >= 8192, n >= 8192, false, true, true, true});
}

bool mmvq_tc_wide(int wt, int64_t k, int64_t m) {
    return wt == GGUF_Q4_K && m > 8 && m <= option_mmvq_tc_max_m() && option_mmvq_tc() && k <= 16384 &&
           mma_q4k_fits(k, m);
}

cudaError_t launch_mmvq_routes_q4_k(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s) {
    return launch_mmvq_routes_pt<Q4KPiece>(bank, rt, n, k, k / 256 * Q4_K_BYTES, xq, routes, z, s);
}

}  // namespace gg
