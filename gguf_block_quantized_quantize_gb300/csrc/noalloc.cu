// gguf_mul_mat_noalloc: the decode-sized mul_mat (m <= 8, the MMVQ path) with
// its q8_1 scratch in a fixed device array owned by this library, for callers
// that cannot get device memory where they call.
//
// The scratch is one array per device and per loaded copy of the library, so
// two calls that overlap in time on the same device (two streams, two host
// threads) race on it.  The first call on a device looks its address up
// (cudaGetSymbolAddress), which must not happen during stream capture: make
// one ordinary call per device first.  The address is kept for the life of
// the process: it is not valid across cudaDeviceReset (the module may load
// elsewhere in the new context), so a process that resets a device must not
// call this entry point on that device afterwards.
#include <stdio.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace gg {

// q8_1 rows of at most 8 x 16384 activation values take 147,456 bytes
constexpr size_t NOALLOC_SCRATCH_BYTES = 256 * 1024;
static __device__ __align__(256) uint8_t g_noalloc_scratch[NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device: the host-side
// symbol is only a stand-in, so the address is looked up once per device.
static gguf_status noalloc_scratch(uint8_t **out) {
    static uint8_t *addr[64] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return report(GGUF_ERR_CUDA, "mul_mat_noalloc: cudaGetDevice failed");
    if (dev < 0 || dev >= 64) return report(GGUF_ERR_INVALID_ARG, "mul_mat_noalloc: device index out of range");
    std::lock_guard<std::mutex> lock(mu);
    if (!addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) {
            char msg[256];
            snprintf(msg, sizeof(msg), "mul_mat_noalloc: scratch address lookup failed (%s)", cudaGetErrorString(e));
            return report(GGUF_ERR_CUDA, msg);
        }
        addr[dev] = (uint8_t *)p;
    }
    *out = addr[dev];
    return GGUF_OK;
}

static bool is_float_t(int t) { return t == GGUF_F32 || t == GGUF_F16 || t == GGUF_BF16; }
static bool is_weight_t(int t) {
    return t == GGUF_Q8_0 || t == GGUF_Q4_0 || t == GGUF_Q4_K || t == GGUF_Q5_K || t == GGUF_Q6_K ||
           t == GGUF_MXFP4;
}
static bool aligned_to(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

}  // namespace gg

using namespace gg;

extern "C" gguf_status gguf_mul_mat_noalloc(const void *w, int wt, int64_t n, int64_t k, const void *x, int xt,
                                            int64_t m, int64_t ldx, void *y, int yt, int64_t ldy,
                                            gguf_stream_t stream) {
    if (!is_weight_t(wt)) return report(GGUF_ERR_UNSUPPORTED_TYPE, "mul_mat_noalloc: weight type not Q8_0/Q4_0/Q4_K/Q5_K/Q6_K/MXFP4");
    if (!is_float_t(xt)) return report(GGUF_ERR_UNSUPPORTED_TYPE, "mul_mat_noalloc: x type is not F32/BF16/F16");
    if (!is_float_t(yt)) return report(GGUF_ERR_UNSUPPORTED_TYPE, "mul_mat_noalloc: y type is not F32/BF16/F16");
    if (n < 0 || k < 0 || m < 0) return report(GGUF_ERR_INVALID_ARG, "mul_mat_noalloc: negative size");
    const int64_t be = block_elems(wt);
    if (k % be) return report(GGUF_ERR_SHAPE, "mul_mat_noalloc: k is not a multiple of the weight block");
    if (ldy < n || ldx < k) return report(GGUF_ERR_INVALID_ARG, "mul_mat_noalloc: ldx < k or ldy < n");
    if (m > 8 || k > 16384)
        return report(GGUF_ERR_WORKSPACE,
                      "mul_mat_noalloc: the fixed scratch serves m <= 8 and k <= 16384 only; use gguf_mul_mat");
    const size_t need = (size_t)m * (size_t)(k / 32) * 36;
    if (need > NOALLOC_SCRATCH_BYTES) return report(GGUF_ERR_WORKSPACE, "mul_mat_noalloc: scratch too small");
    if (m == 0 || n == 0) return GGUF_OK;   // nothing to compute: pointers are not looked at
    if (k == 0) return report(GGUF_ERR_SHAPE, "mul_mat_noalloc: k must be positive");
    if (!w || !x || !y) return report(GGUF_ERR_INVALID_ARG, "mul_mat_noalloc: null pointer");
    const size_t xs = xt == GGUF_F32 ? 4 : 2, ys = yt == GGUF_F32 ? 4 : 2;
    if (!aligned_to(w, 16) || !aligned_to(x, xs) || !aligned_to(y, ys))
        return report(GGUF_ERR_ALIGNMENT, "mul_mat_noalloc: misaligned w, x or y");
    uint8_t *xq = nullptr;
    gguf_status st = noalloc_scratch(&xq);
    if (st != GGUF_OK) return st;
    // the quantize pass overwrites every scratch byte the MMVQ pass reads, so
    // nothing has to be cleared between calls
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = launch_quantize_q8_1(x, xt, m, k, ldx, xq, nullptr, nullptr, s);
    if (e == cudaSuccess) e = launch_mmvq(mmvq_one_segment(w, n, y, ldy), wt, k, xq, m, yt, s);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "mul_mat_noalloc: CUDA error %d (%s)", (int)e, cudaGetErrorString(e));
        return report(GGUF_ERR_CUDA, msg);
    }
    return GGUF_OK;
}
