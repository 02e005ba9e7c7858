// Staging copies between pinned host memory and device memory, run on the SMs
// as a programmatic dependent launch (gguf_copy_async).
//
// A decode step moves a few hundred KB between the host and the GPU.  A
// copy-engine copy of that size costs about 5 us of latency on GB300 and,
// queued between kernels, ends the chain of programmatic dependent launches
// that lets each kernel start while the previous one drains.  Reading or
// writing pinned host memory from a kernel (the unified address space maps it
// for the device; on GB300 the link is NVLink-C2C) keeps the copy inside the
// chain.  Both buffers must be device-accessible: device memory, managed
// memory, or pinned (page-locked) host memory; the ABI entry checks this
// before launching.
#include "common.cuh"
#include "internal.h"

namespace gg {

// dst[0, n) = src[0, n).  V16: both pointers 16-byte aligned, so the bulk
// moves as uint4 words and only a tail of n % 16 bytes is copied byte by byte.
template <bool V16>
__global__ void __launch_bounds__(256) copy_kernel(uint8_t *__restrict__ dst, const uint8_t *__restrict__ src,
                                                   int64_t n) {
    // src may be written, and dst read, by the previous kernel of the stream
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t tid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t nthr = (int64_t)gridDim.x * blockDim.x;
    int64_t done = 0;
    if constexpr (V16) {
        const int64_t nv = n / 16;
        const uint4 *s = reinterpret_cast<const uint4 *>(src);
        uint4 *d = reinterpret_cast<uint4 *>(dst);
        // four independent loads in flight per thread before the stores
        int64_t i = tid;
        for (; i + 3 * nthr < nv; i += 4 * nthr) {
            const uint4 a = s[i], b = s[i + nthr], c = s[i + 2 * nthr], e = s[i + 3 * nthr];
            d[i] = a;
            d[i + nthr] = b;
            d[i + 2 * nthr] = c;
            d[i + 3 * nthr] = e;
        }
        for (; i < nv; i += nthr) d[i] = s[i];
        done = nv * 16;
    }
    for (int64_t i = done + tid; i < n; i += nthr) dst[i] = src[i];
}

cudaError_t launch_copy(void *dst, const void *src, int64_t bytes, cudaStream_t s) {
    if (bytes <= 0) return cudaSuccess;
    const bool v16 = ((reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src)) & 15) == 0;
    const int64_t units = v16 ? (bytes + 15) / 16 : bytes;
    // host memory answers in about a microsecond: enough CTAs that each thread
    // moves two units (one round trip), at most 4 per SM
    int64_t grid = (units + 511) / 512;
    const int64_t cap = (int64_t)device_info().sm_count * 4;
    if (grid > cap) grid = cap;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto *d = reinterpret_cast<uint8_t *>(dst);
    auto *sp = reinterpret_cast<const uint8_t *>(src);
    return v16 ? cudaLaunchKernelEx(&cfg, copy_kernel<true>, d, sp, bytes)
               : cudaLaunchKernelEx(&cfg, copy_kernel<false>, d, sp, bytes);
}

}  // namespace gg
