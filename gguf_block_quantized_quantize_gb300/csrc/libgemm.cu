// The library-GEMM engine of the prefill product: after the weights are
// dequantized to fp16 (dequant.cu) and the activations quantized to q8_1 and
// written as their fp16 operand d16 * q (quantize.cu), the dense product
// y[m][n] = X[m][k] . W[n][k]^T is one cuBLAS GEMM (fp16 operands, fp32
// accumulation; fp16 output directly, other outputs through fp32 rows, since
// the library's fp16-operand GEMM writes fp16 or fp32).  FreeToken PR #196 ("sm_120 dispatch thresholds
// + upstream int8-MMA MMQ port", "Gains" table) races such a dequantize +
// library GEMM path against the fused MMQ on the same shapes; here it is the
// alternative engine of option "mmq_engine" and a cross-check of the fused
// tensor-core MMQ.
//
// cuBLAS is opened at run time (dlopen) on the first use, so the library has no
// link-time dependency on it; without it the engine reports an error and the
// fused MMQ is unaffected.
#include <cublas_v2.h>
#include <dlfcn.h>

#include <mutex>

#include "internal.h"

namespace gg {

namespace {

// the C signature of cublasGemmEx (the C++ header also declares overloads)
using GemmExFn = cublasStatus_t (*)(cublasHandle_t, cublasOperation_t, cublasOperation_t, int, int, int, const void *,
                                    const void *, cudaDataType, int, const void *, cudaDataType, int, const void *,
                                    void *, cudaDataType, int, cublasComputeType_t, cublasGemmAlgo_t);

struct CublasApi {
    decltype(&cublasCreate_v2) create = nullptr;
    decltype(&cublasSetStream_v2) set_stream = nullptr;
    GemmExFn gemm = nullptr;
    bool tried = false, ok = false;
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
CublasApi g_api;
cublasHandle_t g_handle[kMaxDevices] = {};

bool load_api() {
    if (g_api.tried) return g_api.ok;
    g_api.tried = true;
    const char *names[] = {"libcublas.so.13", "libcublas.so", "/usr/local/cuda/lib64/libcublas.so.13"};
    void *h = nullptr;
    for (const char *nm : names)
        if ((h = dlopen(nm, RTLD_NOW | RTLD_GLOBAL)) != nullptr) break;
    if (!h) return false;
    g_api.create = reinterpret_cast<decltype(g_api.create)>(dlsym(h, "cublasCreate_v2"));
    g_api.set_stream = reinterpret_cast<decltype(g_api.set_stream)>(dlsym(h, "cublasSetStream_v2"));
    g_api.gemm = reinterpret_cast<decltype(g_api.gemm)>(dlsym(h, "cublasGemmEx"));
    g_api.ok = g_api.create && g_api.set_stream && g_api.gemm;
    return g_api.ok;
}

}  // namespace

cudaError_t library_gemm_f16(const uint16_t *w, const uint16_t *x, int64_t n, int64_t m, int64_t k, void *y, int yt,
                             int64_t ldy, cudaStream_t s) {
    if (yt != GGUF_F32 && yt != GGUF_F16) return cudaErrorInvalidValue;
    if (n > INT32_MAX || m > INT32_MAX || k > INT32_MAX || ldy > INT32_MAX) return cudaErrorInvalidValue;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cublasHandle_t h;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (!load_api()) return cudaErrorNotSupported;
        if (!g_handle[dev] && g_api.create(&g_handle[dev]) != CUBLAS_STATUS_SUCCESS) {
            g_handle[dev] = nullptr;
            return cudaErrorNotSupported;
        }
        h = g_handle[dev];
    }
    if (g_api.set_stream(h, s) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
    // column-major view: Y^T [n][m] (leading dimension ldy) = W [k][n]^T . X^T [k][m]
    const float alpha = 1.0f, beta = 0.0f;
    const cublasStatus_t st =
        g_api.gemm(h, CUBLAS_OP_T, CUBLAS_OP_N, (int)n, (int)m, (int)k, &alpha, w, CUDA_R_16F, (int)k, x, CUDA_R_16F,
                   (int)k, &beta, y, yt == GGUF_F32 ? CUDA_R_32F : CUDA_R_16F, (int)ldy, CUBLAS_COMPUTE_32F,
                   CUBLAS_GEMM_DEFAULT);
    return st == CUBLAS_STATUS_SUCCESS ? cudaSuccess : cudaErrorUnknown;
}

}  // namespace gg
