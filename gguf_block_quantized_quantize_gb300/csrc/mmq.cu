// MMQ: tensor-core product of packed weights with many activation rows
// (prefill).  y[m][n] = sum_k W[n][k] * Xq[m][k] where Xq is the q8_1
// quantization of the activations.
//
// The pages' MMQ (FreeToken PR #196 "sm_120 dispatch thresholds + upstream
// int8-MMA MMQ port", section "What") contracts int8 quants on int8 tensor-core
// tiles and scales each 32-block result on CUDA cores.  sm_103a has no int8
// tcgen05 MMA (ptxas rejects tcgen05.mma.kind::i8 for sm_103a), and a per-block
// rescale read out of TMEM every 32 (Q6_K: 16) values would cost more FP32 work
// than the tensor core does.  This kernel therefore feeds tcgen05.mma.kind::f16
// with fp16 operands that hold the dequantized values -- the weight unpacked in
// registers (fp32 value of the block formula, rounded once to fp16) and the
// q8_1 activation d16 * q (rounded once to fp16, written by the quantize pass)
// -- and accumulates over the whole K in fp32 in TMEM.  Every per-block scale
// and min of the blockwise formula is applied exactly in fp32 before the
// single fp16 rounding, so the result differs from the fp64 blockwise formula
// only by those two roundings (about 3e-4 of the row rms).
//
// Tile: 128 weight rows (UMMA M) x BN activation rows (UMMA N) x 64 K per stage,
// 4 stages.  Roles (192 threads):
//   warp 0   : TMA producer of the activation tile (128-byte swizzle)
//   warp 1   : TMEM allocator and the single MMA-issuing thread
//   warps 2-5: weight producers (one weight row per thread: packed bytes are
//              prefetched two K-steps ahead, unpacked to fp16 and stored in the
//              128-byte-swizzled K-major layout), then the epilogue (TMEM ->
//              registers -> y in the output dtype).
// Every wait is bounded (1 s); a timeout sets *err and the CTA exits cleanly.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "unpack.cuh"

namespace gg {

constexpr int MMQ_BM = 128;
constexpr int MMQ_BK = 64;
constexpr int MMQ_STAGES = 4;
constexpr int MMQ_THREADS = 192;
constexpr int MMQ_A_BYTES = MMQ_BM * MMQ_BK * 2;  // 16 KB

__device__ int g_mmq_error;  // nonzero after a timed-out wait (diagnostics)

__host__ __device__ constexpr int mmq_b_bytes(int bn) { return bn * MMQ_BK * 2; }
__host__ __device__ constexpr int mmq_tmem_cols(int bn) { return bn < 32 ? 32 : bn; }
__host__ __device__ constexpr int mmq_smem_bytes(int bn) {
    return 1024 /* alignment slack */ + MMQ_STAGES * (MMQ_A_BYTES + mmq_b_bytes(bn)) + 256 /* barriers */;
}

template <int WT, int BN, int OT>
__global__ void __launch_bounds__(MMQ_THREADS, 1)
    mmq_kernel(const __grid_constant__ CUtensorMap tmap_x, const uint8_t *__restrict__ w, int64_t n, int64_t k,
               int64_t rb, int64_t m, void *__restrict__ y, int64_t ldy) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + MMQ_STAGES * MMQ_A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + MMQ_STAGES * mmq_b_bytes(BN));
    uint64_t *full_a = bars;                    // 128 weight-producer arrivals
    uint64_t *full_b = bars + MMQ_STAGES;       // TMA bytes
    uint64_t *empty = bars + 2 * MMQ_STAGES;    // MMA commit
    uint64_t *done = bars + 3 * MMQ_STAGES;     // last MMA commit
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * MMQ_STAGES + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int64_t n0 = (int64_t)blockIdx.x * MMQ_BM;
    const int64_t m0 = (int64_t)blockIdx.y * BN;
    const int KS = (int)((k + MMQ_BK - 1) / MMQ_BK);
    constexpr uint32_t TMEM_COLS = mmq_tmem_cols(BN);

    if (tid == 0) {
        for (int s = 0; s < MMQ_STAGES; s++) {
            tc::mbar_init(&full_a[s], 128);
            tc::mbar_init(&full_b[s], 1);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(done, 1);
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::prefetch_tmap(&tmap_x);
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    auto fail = [&](int code) {
        *abort_flag = 1;
        atomicOr(&g_mmq_error, code);
    };

    if (warp == 0) {
        // ---------------- TMA producer (activation tiles)
        if (lane == 0) {
            int issued = 0;
            for (int ks = 0; ks < KS; ks++) {
                const int s = ks % MMQ_STAGES;
                const uint32_t ph = (uint32_t)(ks / MMQ_STAGES) & 1u;
                if (*abort_flag) break;
                if (!tc::mbar_wait(&empty[s], ph ^ 1u)) { fail(1); break; }
                tc::mbar_arrive_expect_tx(&full_b[s], (uint32_t)mmq_b_bytes(BN));
                tc::tma_load_2d(sB + s * mmq_b_bytes(BN), &tmap_x, &full_b[s], ks * MMQ_BK, (int32_t)m0);
                issued = ks + 1;
            }
            // on abort, let the copies already issued land before the CTA exits
            if (*abort_flag) {
                for (int ks = issued - MMQ_STAGES < 0 ? 0 : issued - MMQ_STAGES; ks < issued; ks++)
                    tc::mbar_wait(&full_b[ks % MMQ_STAGES], (uint32_t)(ks / MMQ_STAGES) & 1u);
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = tc::idesc_f16_f32(MMQ_BM, BN);
            for (int ks = 0; ks < KS; ks++) {
                const int s = ks % MMQ_STAGES;
                const uint32_t ph = (uint32_t)(ks / MMQ_STAGES) & 1u;
                if (*abort_flag) break;
                if (!tc::mbar_wait(&full_a[s], ph) || !tc::mbar_wait(&full_b[s], ph)) { fail(2); break; }
                tc::tc_fence_after();
                const uint32_t a0 = tc::smem_u32(sA + s * MMQ_A_BYTES);
                const uint32_t b0 = tc::smem_u32(sB + s * mmq_b_bytes(BN));
#pragma unroll
                for (int kk = 0; kk < MMQ_BK / 16; kk++) {
                    tc::mma_f16(tmem, tc::sw128_desc(a0 + 32 * kk), tc::sw128_desc(b0 + 32 * kk), idesc,
                                (ks | kk) != 0 ? 1u : 0u);
                }
                tc::mma_commit(&empty[s]);
            }
            tc::mma_commit(done);  // arrives once every MMA issued above has completed
        }
    } else {
        // ---------------- weight producers, then the epilogue
        const int t = tid - 64;  // weight row within the tile
        const int64_t row = n0 + t;
        const bool live = row < n;
        const uint8_t *wrow = w + (live ? row : 0) * rb;
        KUnit<WT> u[2];
        if constexpr (WT == GGUF_Q8_0) { u[0].kblocks = k / 32; u[1].kblocks = k / 32; }
        if (live) {
            u[0].load(wrow, 0);
            if (KS > 1) u[1].load(wrow, 1);
        }
        for (int ks0 = 0; ks0 < KS; ks0 += 2) {
#pragma unroll
            for (int j = 0; j < 2; j++) {
                const int ks = ks0 + j;
                if (ks >= KS) break;
                const int s = ks % MMQ_STAGES;
                const uint32_t ph = (uint32_t)(ks / MMQ_STAGES) & 1u;
                uint32_t vals[32];
                if (live) u[j].unpack(ks, vals);
                else {
#pragma unroll
                    for (int i = 0; i < 32; i++) vals[i] = 0u;
                }
                if (live && ks + 2 < KS) u[j].load(wrow, ks + 2);  // prefetch two K-steps ahead
                if (*abort_flag) break;
                if (!tc::mbar_wait(&empty[s], ph ^ 1u)) { fail(4); break; }
                store_sw128_row(sA + s * MMQ_A_BYTES, t, vals);
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(&full_a[s]);
            }
            if (*abort_flag) break;
        }
        // ---------------- epilogue: TMEM lane quadrant (warp % 4) -> rows
        const bool ok = tc::mbar_wait(done, 0);
        if (!ok) fail(8);
        tc::tc_fence_after();
        if (ok && !*abort_flag) {
            const int q = warp & 3;
            const int64_t orow = n0 + 32 * q + lane;
#pragma unroll 1
            for (int c = 0; c < BN / 32 || (BN < 32 && c == 0); c++) {
                uint32_t r[32];
                tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + 32 * c, r);
                tc::tmem_ld_wait();
                if (orow < n) {
#pragma unroll
                    for (int jj = 0; jj < 32; jj++) {
                        const int64_t mm = m0 + 32 * c + jj;
                        if (jj < BN && mm < m) store_out(y, OT, mm * ldy + orow, __uint_as_float(r[jj]));
                    }
                }
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// ---------------------------------------------------------------- host side

static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// fp16 activation rows [m][k] as a TMA tensor map with a 64 x bn box
static cudaError_t make_x_map(CUtensorMap *map, const uint16_t *xh, int64_t m, int64_t k, int bn) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t gdim[2] = {(cuuint64_t)k, (cuuint64_t)m};
    cuuint64_t gstride[1] = {(cuuint64_t)k * 2};
    cuuint32_t box[2] = {(cuuint32_t)MMQ_BK, (cuuint32_t)bn};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(xh), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int WT, int BN, int OT>
static cudaError_t launch_mmq_t(const uint8_t *w, int64_t n, int64_t k, const uint16_t *xh, int64_t m, void *y,
                                int64_t ldy, cudaStream_t s) {
    CUtensorMap map;
    cudaError_t e = make_x_map(&map, xh, m, k, BN);
    if (e != cudaSuccess) return e;
    auto kern = mmq_kernel<WT, BN, OT>;
    constexpr int smem = mmq_smem_bytes(BN);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    const int64_t rb = k / block_elems(WT) * block_bytes(WT);
    dim3 grid((unsigned)((n + MMQ_BM - 1) / MMQ_BM), (unsigned)((m + BN - 1) / BN));
    kern<<<grid, MMQ_THREADS, smem, s>>>(map, w, n, k, rb, m, y, ldy);
    return cudaGetLastError();
}

template <int WT, int OT>
static cudaError_t launch_mmq_bn(const uint8_t *w, int64_t n, int64_t k, const uint16_t *xh, int64_t m, void *y,
                                 int64_t ldy, cudaStream_t s) {
    if (m <= 16) return launch_mmq_t<WT, 16, OT>(w, n, k, xh, m, y, ldy, s);
    if (m <= 32) return launch_mmq_t<WT, 32, OT>(w, n, k, xh, m, y, ldy, s);
    if (m <= 64) return launch_mmq_t<WT, 64, OT>(w, n, k, xh, m, y, ldy, s);
    if (m <= 128) return launch_mmq_t<WT, 128, OT>(w, n, k, xh, m, y, ldy, s);
    return launch_mmq_t<WT, 256, OT>(w, n, k, xh, m, y, ldy, s);
}

template <int WT>
static cudaError_t launch_mmq_ot(const uint8_t *w, int64_t n, int64_t k, const uint16_t *xh, int64_t m, void *y,
                                 int yt, int64_t ldy, cudaStream_t s) {
    if (yt == GGUF_F32) return launch_mmq_bn<WT, GGUF_F32>(w, n, k, xh, m, y, ldy, s);
    if (yt == GGUF_BF16) return launch_mmq_bn<WT, GGUF_BF16>(w, n, k, xh, m, y, ldy, s);
    return launch_mmq_bn<WT, GGUF_F16>(w, n, k, xh, m, y, ldy, s);
}

cudaError_t launch_mmq(const uint8_t *w, int wt, int64_t n, int64_t k, const uint16_t *xh, int64_t m, void *y,
                       int yt, int64_t ldy, cudaStream_t s) {
    if (n == 0 || m == 0) return cudaSuccess;
    if ((reinterpret_cast<uintptr_t>(xh) & 15) || (k % 8)) return cudaErrorInvalidValue;
    switch (wt) {
    case GGUF_Q4_K: return launch_mmq_ot<GGUF_Q4_K>(w, n, k, xh, m, y, yt, ldy, s);
    case GGUF_Q6_K: return launch_mmq_ot<GGUF_Q6_K>(w, n, k, xh, m, y, yt, ldy, s);
    case GGUF_Q8_0: return launch_mmq_ot<GGUF_Q8_0>(w, n, k, xh, m, y, yt, ldy, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace gg
