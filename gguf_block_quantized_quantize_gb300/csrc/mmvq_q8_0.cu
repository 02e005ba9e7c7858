// MMVQ instantiations for Q8_0 weights (see mmvq.cuh).
#include "mmvq.cuh"

namespace gg {

cudaError_t launch_mmvq_q8_0(const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, void *y, int yt,
                             int64_t ldy, cudaStream_t s) {
    return launch_mmvq_pt<ThinPiece<GGUF_Q8_0>>(w, n, k, xq, m, y, yt, ldy, s, k / 32 * Q8_0_BYTES, MmvqTune{false, false, true});
}

}  // namespace gg
