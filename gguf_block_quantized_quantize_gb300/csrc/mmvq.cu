// MMVQ dispatch by weight type (kernels in mmvq.cuh, one translation unit per type).
#include "mmvq.cuh"

namespace gg {

// One piece per thread and at most 512 threads per CTA: K <= 16384 (longer
// rows take the tensor-core path, which has no K limit).
constexpr int64_t MMVQ_MAX_PIECES = 512;

MmvqSegs mmvq_one_segment(const void *w, int64_t n, void *y, int64_t ldy) {
    MmvqSegs sg{};
    sg.nseg = 1;
    for (int i = 0; i < MMVQ_MAX_SEGS; i++) sg.end[i] = INT64_MAX;
    sg.end[0] = n;
    sg.w[0] = (const uint8_t *)w;
    sg.y[0] = y;
    sg.ldy[0] = ldy;
    return sg;
}

cudaError_t launch_mmvq(const MmvqSegs &sg, int wt, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s) {
    if (sg.nseg < 1 || sg.nseg > MMVQ_MAX_SEGS) return cudaErrorInvalidValue;
    if (sg.rows() == 0 || m == 0) return cudaSuccess;
    if (k / 32 > MMVQ_MAX_PIECES || (m > 8 && !mmvq_tc_wide(wt, k, m))) return cudaErrorInvalidValue;
    switch (wt) {
    case GGUF_Q8_0: return launch_mmvq_q8_0(sg, k, xq, m, yt, s);
    case GGUF_Q4_K: return launch_mmvq_q4_k(sg, k, xq, m, yt, s);
    case GGUF_Q6_K: return launch_mmvq_q6_k(sg, k, xq, m, yt, s);
    case GGUF_Q4_0: return launch_mmvq_q4_0(sg, k, xq, m, yt, s);
    case GGUF_Q5_K: return launch_mmvq_q5_k(sg, k, xq, m, yt, s);
    case GGUF_MXFP4: return launch_mmvq_mxfp4(sg, k, xq, m, yt, s);
    default: return cudaErrorInvalidValue;
    }
}

__global__ void mmvq_join_kernel() {}

// an ordinary (non-programmatic) launch: it starts only after all earlier work
// of the stream has completed, which closes a batch of chained MMVQ launches
cudaError_t launch_mmvq_join(cudaStream_t s) {
    mmvq_join_kernel<<<1, 32, 0, s>>>();
    return cudaGetLastError();
}

bool mmvq_routes_supported(int wt, int64_t k) {
    const int64_t values = wt == GGUF_Q8_0 ? 32 : 64;   // values per thread's piece
    return (wt == GGUF_Q8_0 || wt == GGUF_Q4_0 || wt == GGUF_Q4_K || wt == GGUF_Q5_K || wt == GGUF_Q6_K ||
            wt == GGUF_MXFP4) && k > 0 && (k + values - 1) / values <= 256;
}

cudaError_t launch_mmvq_routes(int wt, const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k,
                               const uint8_t *xq, int64_t routes, float *z, cudaStream_t s) {
    if (!mmvq_routes_supported(wt, k)) return cudaErrorInvalidValue;
    switch (wt) {
    case GGUF_Q8_0: return launch_mmvq_routes_q8_0(bank, rt, n, k, xq, routes, z, s);
    case GGUF_Q4_K: return launch_mmvq_routes_q4_k(bank, rt, n, k, xq, routes, z, s);
    case GGUF_Q4_0: return launch_mmvq_routes_q4_0(bank, rt, n, k, xq, routes, z, s);
    case GGUF_Q5_K: return launch_mmvq_routes_q5_k(bank, rt, n, k, xq, routes, z, s);
    case GGUF_MXFP4: return launch_mmvq_routes_mxfp4(bank, rt, n, k, xq, routes, z, s);
    default: return launch_mmvq_routes_q6_k(bank, rt, n, k, xq, routes, z, s);
    }
}

}  // namespace gg
