// MMQ: tensor-core product of packed weights with many activation rows
// (prefill), y[m][n] = sum_k W[n][k] * Xq[m][k], Xq the q8_1 activations.
//
// The pages' MMQ (FreeToken PR #196 "sm_120 dispatch thresholds + upstream
// int8-MMA MMQ port", section "What") contracts int8 quants on int8 tensor-core
// tiles and scales each 32-block result on CUDA cores.  sm_103a has no int8
// tcgen05 MMA (ptxas rejects tcgen05.mma.kind::i8 for sm_103a), and a per-block
// rescale read out of TMEM every 32 (Q6_K: 16) values would cost more FP32 work
// than the tensor core does.  This path therefore feeds tcgen05.mma.kind::f16
// with fp16 operands holding the dequantized values -- every per-block scale
// and min applied exactly in fp32 first -- and accumulates over K in fp32 in
// TMEM (tcgemm.cuh).  16-bit outputs use one fp16 operand per side; fp32
// outputs use the hi + lo split on both sides (three MMAs per K step), which
// matches the exact blockwise value to about 1e-6.
//
// Tiles of 128 weight rows x BN activation rows, persistent over the GPU; small
// token counts split K across CTAs (fp32 partial sums in the workspace, then a
// conversion pass) so that every SM has work.
#include <stdio.h>

#include <mutex>

#include "tcgemm.cuh"

namespace gg {

// Error word of the tensor-core kernels: a CTA whose bounded wait gives up ORs
// in the bit of its role (1 operand-B loads, 2 MMA issue, 4 weight unpack,
// 8 epilogue, 16 accumulator hand-over, 32 packed-weight loads) and exits.
// gguf_device_errors reads it back.
__device__ int g_tg_error;

int *tg_error_word() {
    static int *ptr[64] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptr[dev] && cudaGetSymbolAddress(reinterpret_cast<void **>(&ptr[dev]), g_tg_error) != cudaSuccess)
        ptr[dev] = nullptr;
    return ptr[dev];
}

// *dst = the error word (stream-ordered); clear: reset it to 0 in the same step
__global__ void tg_error_take_kernel(int32_t *dst, int clear) {
    *dst = clear ? atomicExch(&g_tg_error, 0) : atomicOr(&g_tg_error, 0);
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

template <int WT, int BN, bool PRECISE, int OT>
static cudaError_t launch_dense(const uint8_t *w, int64_t n, int64_t k, const uint16_t *xh, const uint16_t *xl,
                                int64_t m, void *y, int64_t ldy, float *yacc, cudaStream_t s) {
    const int64_t kx = op_pitch(WT, k);
    CUtensorMap mh, ml, mw;
    cudaError_t e = tg_make_map(&mh, xh, m, kx, BN);
    if (e != cudaSuccess) return e;
    ml = mh;
    mw = mh;
    if (PRECISE && (e = tg_make_map(&ml, xl, m, kx, BN)) != cudaSuccess) return e;
    TgParams p{};
    p.w = w;
    p.rb = k / block_elems(WT) * block_bytes(WT);
    p.n = n;
    p.k = k;
    p.kx = kx;
    p.m = m;
    if (option_mmq_stage())
        tg_plan_staging(p, &mw, WT, w, n, 1, 0, k, TG_BM, tg_base_bytes<WT, BN, PRECISE, TG_DENSE>());
    const int64_t tiles_n = (n + TG_BM - 1) / TG_BM, tiles_m = (m + BN - 1) / BN;
    const int KS = (int)((kx + TG_BK - 1) / TG_BK);
    const int sms = device_info().sm_count;
    int splits = 1;
    if (yacc != nullptr) {  // split K until the tiles fill the GPU, keeping >= 4 K-steps per split
        const int64_t base = tiles_n * tiles_m;
        while (base * splits < sms && (KS + splits) / (splits + 1) >= 4) splits++;
    }
    int kps = (KS + splits - 1) / splits;
    if (p.pstages > 0 && p.pchunked) kps = (kps + 3) / 4 * 4;   // splits start on a staged chunk
    splits = (KS + kps - 1) / kps;
    const int64_t tiles = tiles_n * tiles_m * splits;
    if (tiles > INT32_MAX) return cudaErrorInvalidValue;
    p.tiles_n = (int)tiles_n;
    p.tiles_m = (int)tiles_m;
    // weights that do not stay in L2 across a pass over the weight tiles (the
    // LM head: 417 MB of Q6_K) are read once per activation tile in the
    // weight-fastest order; activation-fastest reads each once
    p.m_fast = (tiles_m > 1 && n * p.rb > (int64_t)(64 << 20)) ? 1 : 0;
    p.tiles_total = (int)tiles;
    p.ks_per_split = kps;
    p.y = y;
    p.yt = OT;
    p.ldy = ldy;
    p.yacc = splits > 1 ? yacc : nullptr;
    if (splits > 1 && (e = cudaMemsetAsync(yacc, 0, sizeof(float) * (size_t)(m * n), s)) != cudaSuccess) return e;
    CUtensorMap my = mh;
    p.ystore = (splits == 1 && tg_make_out_map(&my, y, OT, n, m, ldy)) ? 1 : 0;
    const int grid = (int)(tiles < sms ? tiles : sms);
    e = tg_launch<WT, BN, PRECISE, TG_DENSE, OT>(mh, ml, mw, my, p, grid, s);
    if (e != cudaSuccess || splits == 1) return e;
    return launch_convert_rows(yacc, m, n, y, OT, ldy, s);
}

template <int WT, int OT>
static cudaError_t launch_mmq_bn(const uint8_t *w, int64_t n, int64_t k, const uint16_t *xh, const uint16_t *xl,
                                 int64_t m, void *y, int64_t ldy, float *yacc, cudaStream_t s) {
    if constexpr (OT == GGUF_F32) {  // precise: hi + lo operands
        if (m <= 32) return launch_dense<WT, 32, true, OT>(w, n, k, xh, xl, m, y, ldy, yacc, s);
        if (m <= 64) return launch_dense<WT, 64, true, OT>(w, n, k, xh, xl, m, y, ldy, yacc, s);
        return launch_dense<WT, 128, true, OT>(w, n, k, xh, xl, m, y, ldy, yacc, s);
    } else {
    if (m <= 16) return launch_dense<WT, 16, false, OT>(w, n, k, xh, xl, m, y, ldy, yacc, s);
    if (m <= 32) return launch_dense<WT, 32, false, OT>(w, n, k, xh, xl, m, y, ldy, yacc, s);
    if (m <= 64) return launch_dense<WT, 64, false, OT>(w, n, k, xh, xl, m, y, ldy, yacc, s);
    if (m <= 128 || option_mmq_bn_max() <= 128) return launch_dense<WT, 128, false, OT>(w, n, k, xh, xl, m, y, ldy, yacc, s);
    return launch_dense<WT, 256, false, OT>(w, n, k, xh, xl, m, y, ldy, yacc, s);
    }
}

template <int WT>
static cudaError_t launch_mmq_ot(const uint8_t *w, int64_t n, int64_t k, const uint16_t *xh, const uint16_t *xl,
                                 int64_t m, void *y, int yt, int64_t ldy, float *yacc, cudaStream_t s) {
    if (yt == GGUF_F32) return launch_mmq_bn<WT, GGUF_F32>(w, n, k, xh, xl, m, y, ldy, yacc, s);
    if (yt == GGUF_BF16) return launch_mmq_bn<WT, GGUF_BF16>(w, n, k, xh, xl, m, y, ldy, yacc, s);
    return launch_mmq_bn<WT, GGUF_F16>(w, n, k, xh, xl, m, y, ldy, yacc, s);
}

cudaError_t launch_mmq(const uint8_t *w, int wt, int64_t n, int64_t k, const uint16_t *xh, const uint16_t *xl,
                       int64_t m, void *y, int yt, int64_t ldy, float *yacc, cudaStream_t s) {
    if (n == 0 || m == 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(xh) & 15) || (k % 8)) return cudaErrorInvalidValue;
    if (yt == GGUF_F32 && (xl == nullptr || (reinterpret_cast<uintptr_t>(xl) & 15))) return cudaErrorInvalidValue;
    switch (wt) {
    case GGUF_Q4_K: return launch_mmq_ot<GGUF_Q4_K>(w, n, k, xh, xl, m, y, yt, ldy, yacc, s);
    case GGUF_Q6_K: return launch_mmq_ot<GGUF_Q6_K>(w, n, k, xh, xl, m, y, yt, ldy, yacc, s);
    case GGUF_Q8_0: return launch_mmq_ot<GGUF_Q8_0>(w, n, k, xh, xl, m, y, yt, ldy, yacc, s);
    case GGUF_Q4_0: return launch_mmq_ot<GGUF_Q4_0>(w, n, k, xh, xl, m, y, yt, ldy, yacc, s);
    case GGUF_Q5_K: return launch_mmq_ot<GGUF_Q5_K>(w, n, k, xh, xl, m, y, yt, ldy, yacc, s);
    case GGUF_MXFP4: return launch_mmq_ot<GGUF_MXFP4>(w, n, k, xh, xl, m, y, yt, ldy, yacc, s);
    default: return cudaErrorInvalidValue;
    }
}

// y[m][ldy] (out dtype) from yacc[m][n] fp32
__global__ void convert_rows_kernel(const float *__restrict__ yacc, int64_t m, int64_t n, void *__restrict__ y, int yt,
                                    int64_t ldy) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= m * n) return;
    const int64_t r = i / n, c = i - r * n;
    store_out(y, yt, r * ldy + c, yacc[i]);
}

cudaError_t launch_convert_rows(const float *yacc, int64_t m, int64_t n, void *y, int yt, int64_t ldy, cudaStream_t s) {
    const int64_t total = m * n;
    if (total == 0) return cudaSuccess;
    convert_rows_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(yacc, m, n, y, yt, ldy);
    return cudaGetLastError();
}

}  // namespace gg

using namespace gg;

static gguf_status device_error_status(int v) {
    if (v == 0) return GGUF_OK;
    char msg[256];
    snprintf(msg, sizeof(msg),
             "device_errors: a tensor-core kernel gave up a bounded wait (flags 0x%x:%s%s%s%s%s%s); outputs of "
             "the calls since the last check are not valid",
             v, (v & 1) ? " operand loads" : "", (v & 2) ? " MMA issue" : "", (v & 4) ? " weight unpack" : "",
             (v & 8) ? " epilogue" : "", (v & 16) ? " accumulator hand-over" : "", (v & 32) ? " packed-weight loads" : "");
    return report(GGUF_ERR_DEVICE, msg);
}

extern "C" gguf_status gguf_device_errors(int32_t *flags, int clear, gguf_stream_t stream) {
    if (!flags) return report(GGUF_ERR_INVALID_ARG, "device_errors: null flags");
    *flags = 0;
    int *word = tg_error_word();
    if (!word) return report(GGUF_ERR_CUDA, "device_errors: the error word of the current device is not reachable");
    cudaStream_t s = (cudaStream_t)stream;
    int v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, word, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && clear) e = cudaMemsetAsync(word, 0, sizeof(int), s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "device_errors: CUDA error %d (%s)", (int)e, cudaGetErrorString(e));
        return report(GGUF_ERR_CUDA, msg);
    }
    *flags = v;
    return device_error_status(v);
}

extern "C" gguf_status gguf_device_errors_async(int32_t *dev_flags, int clear, gguf_stream_t stream) {
    if (!dev_flags) return report(GGUF_ERR_INVALID_ARG, "device_errors_async: null flags");
    if (reinterpret_cast<uintptr_t>(dev_flags) % 4) return report(GGUF_ERR_ALIGNMENT, "device_errors_async: flags must be 4-byte aligned");
    tg_error_take_kernel<<<1, 1, 0, (cudaStream_t)stream>>>(dev_flags, clear ? 1 : 0);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char msg[256];
        snprintf(msg, sizeof(msg), "device_errors_async: CUDA error %d (%s)", (int)e, cudaGetErrorString(e));
        return report(GGUF_ERR_CUDA, msg);
    }
    return GGUF_OK;
}
