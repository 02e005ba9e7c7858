// MoE mul_mat_id on the tensor cores, with no host synchronization.
//
// FreeToken PR #690 "serve GGUF checkpoints on vendored ggml-cuda kernels"
// (section "Vendored ggml") launches MoE MMQ only over the (expert, column
// tile) pairs that received routes, so the host never waits for the route
// counts; its op list has the fused GLU and the MoE weighted sum.  FreeToken issue #671
// ("Known issues") records that a token naming the same expert twice, or an
// inactive slot, crashed the prior-art kernel; here both are ordinary routes.
//
// Device-side grouping (three small kernels, all stream-ordered):
//   count   : per route r = t*top_k + j with a valid id e, pos[r] = the r-th
//             slot of expert e (atomic), counts[e]++; ids >= E are counted in
//             the caller's status word; inactive routes get pos = -1.
//   scan    : offsets = exclusive scan of counts; each expert's routes form
//             ceil(count / BN) work tiles; tile (expert, first slot) list and
//             the tile count are written for the GEMM.
//   scatter : route_list[offsets[e] + pos[r]] = r.
// The GEMM is launched with an upper bound of tiles (routes / BN + experts);
// CTAs past the device-side tile count exit at once.
//
// GEMM tile: 128 weight rows x BN routes x 64 K per stage (4 stages), the same
// fp16 tcgen05 engine as the dense MMQ.  The activation rows of a tile are
// gathered with cp.async (token rows for gate_up, route rows for down); the
// last tile of an expert issues the MMA with N rounded up to 16 only.
//   gate_up : the A tile holds 64 gate rows i and the 64 matching up rows I+i,
//             so the epilogue has g and u of the same (route, i): it computes
//             h = silu(g) * u in fp32, rounds it to bf16 (the activation dtype),
//             quantizes each 32 consecutive i (one warp) to a q8_1 block, and
//             writes q8_1 / bf16 / fp16 (d16*q, the operand of the down GEMM).
//   down    : y_acc[t][n] += route_w * (W_down[e] . h_route) with fp32 atomics;
//             a last pass converts y_acc to the output dtype.
#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "unpack.cuh"

namespace gg {

constexpr int MOE_BM = 128;
constexpr int MOE_BK = 64;
constexpr int MOE_STAGES = 4;
constexpr int MOE_THREADS = 192;
constexpr int MOE_A_BYTES = MOE_BM * MOE_BK * 2;
constexpr int MOE_GATHER_LAG = 2;  // cp.async groups in flight per gather lane

__device__ int g_moe_error;

__host__ __device__ constexpr int moe_b_bytes(int bn) { return bn * MOE_BK * 2; }
__host__ __device__ constexpr int moe_smem_bytes(int bn) {
    return 1024 + MOE_STAGES * (MOE_A_BYTES + moe_b_bytes(bn)) + 256 + bn * 8;
}

// ---------------------------------------------------------------- grouping

__global__ void moe_count_kernel(const int32_t *__restrict__ ids, const float *__restrict__ rw, int64_t R,
                                 int64_t E, int skip_zero_w, int32_t *__restrict__ counts, int32_t *__restrict__ pos,
                                 int32_t *__restrict__ dev_status) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= R) return;
    const int32_t e = ids[r];
    const bool ok = e >= 0 && e < E && !(skip_zero_w && rw != nullptr && rw[r] == 0.0f);
    if (e >= E && dev_status != nullptr) atomicAdd(dev_status, 1);
    pos[r] = ok ? atomicAdd(&counts[e], 1) : -1;
}

// single CTA of 1024 threads: exclusive scans of counts and of tiles per expert
__global__ void __launch_bounds__(1024) moe_scan_kernel(const int32_t *__restrict__ counts, int64_t E, int bn,
                                                        int32_t *__restrict__ offsets,
                                                        int32_t *__restrict__ tile_expert,
                                                        int32_t *__restrict__ tile_start,
                                                        int32_t *__restrict__ n_tiles) {
    __shared__ int32_t wsum_c[32], wsum_t[32];
    __shared__ int32_t carry_c, carry_t;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) { carry_c = 0; carry_t = 0; }
    __syncthreads();
    for (int64_t base = 0; base < E; base += 1024) {
        const int64_t e = base + tid;
        const int32_t c = e < E ? counts[e] : 0;
        const int32_t t = (c + bn - 1) / bn;
        int32_t ic = c, it = t;  // inclusive warp scans
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t vc = __shfl_up_sync(0xffffffffu, ic, o), vt = __shfl_up_sync(0xffffffffu, it, o);
            if (lane >= o) { ic += vc; it += vt; }
        }
        if (lane == 31) { wsum_c[warp] = ic; wsum_t[warp] = it; }
        __syncthreads();
        if (warp == 0) {
            int32_t sc = wsum_c[lane], st = wsum_t[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t vc = __shfl_up_sync(0xffffffffu, sc, o), vt = __shfl_up_sync(0xffffffffu, st, o);
                if (lane >= o) { sc += vc; st += vt; }
            }
            wsum_c[lane] = sc - wsum_c[lane];  // exclusive warp offsets
            wsum_t[lane] = st - wsum_t[lane];
        }
        __syncthreads();
        const int32_t ex_c = carry_c + wsum_c[warp] + ic - c;
        const int32_t ex_t = carry_t + wsum_t[warp] + it - t;
        if (e < E) {
            offsets[e] = ex_c;
            for (int32_t i = 0; i < t; i++) {
                tile_expert[ex_t + i] = (int32_t)e;
                tile_start[ex_t + i] = i * bn;
            }
        }
        __syncthreads();
        if (tid == 1023) { carry_c = ex_c + c; carry_t = ex_t + t; }
        __syncthreads();
    }
    if (tid == 0) { offsets[E] = carry_c; *n_tiles = carry_t; }
}

__global__ void moe_scatter_kernel(const int32_t *__restrict__ ids, const int32_t *__restrict__ pos, int64_t R,
                                   const int32_t *__restrict__ offsets, int32_t *__restrict__ route_list) {
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= R) return;
    const int32_t p = pos[r];
    if (p >= 0) route_list[offsets[ids[r]] + p] = (int32_t)r;
}

// ---------------------------------------------------------------- GEMM

enum { MOE_GATE_UP = 0, MOE_DOWN = 1 };

struct MoeParams {
    const uint8_t *w;
    int64_t expert_stride, rb, n, k;
    const uint16_t *xh;       // gather source rows, fp16 [rows][k]
    int64_t top_k;            // gate_up: source row = route / top_k; down: source row = route
    const int32_t *route_list, *offsets, *counts, *tile_expert, *tile_start, *n_tiles;
    const float *route_w;
    uint8_t *hq;              // gate_up outputs (any may be null)
    uint16_t *hbf, *h16;
    float *yacc;              // down output accumulator [T][n]
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <int WT, int BN, int MODE>
__global__ void __launch_bounds__(MOE_THREADS, 1) moe_mmq_kernel(const MoeParams p) {
    const int tile = blockIdx.y;
    if (tile >= *p.n_tiles) return;  // upper-bound grid: nothing routed here
    const int e = p.tile_expert[tile];
    const int s0 = p.tile_start[tile];
    const int cnt = p.counts[e];
    const int n_eff = cnt - s0 < BN ? cnt - s0 : BN;
    const int route0 = p.offsets[e] + s0;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;
    uint8_t *sB = smem + MOE_STAGES * MOE_A_BYTES;
    uint64_t *bars = reinterpret_cast<uint64_t *>(sB + MOE_STAGES * moe_b_bytes(BN));
    uint64_t *full_a = bars, *full_b = bars + MOE_STAGES, *empty = bars + 2 * MOE_STAGES, *done = bars + 3 * MOE_STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * MOE_STAGES + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int32_t *s_route = reinterpret_cast<int32_t *>(bars + 32);   // BN route ids of this tile
    float *s_w = reinterpret_cast<float *>(s_route + BN);         // their weights (down)

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int KS = (int)((p.k + MOE_BK - 1) / MOE_BK);
    constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;

    if (tid == 0) {
        for (int s = 0; s < MOE_STAGES; s++) {
            tc::mbar_init(&full_a[s], 128);
            tc::mbar_init(&full_b[s], 32);
            tc::mbar_init(&empty[s], 1);
        }
        tc::mbar_init(done, 1);
        *abort_flag = 0;
        tc::fence_barrier_init();
    }
    for (int j = tid; j < BN; j += MOE_THREADS) {
        const int r = j < n_eff ? p.route_list[route0 + j] : -1;
        s_route[j] = r;
        if (MODE == MOE_DOWN) s_w[j] = (r >= 0 && p.route_w != nullptr) ? p.route_w[r] : 1.0f;
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
        atomicOr(&g_moe_error, code);
    };

    if (warp == 0) {
        // ---------------- gather producer: BN activation rows per stage, 16-byte cp.async
        constexpr int RPL = (BN + 31) / 32;  // rows per lane
        const uint16_t *src[RPL];
#pragma unroll
        for (int i = 0; i < RPL; i++) {
            const int j = lane + 32 * i;
            const int r = j < BN ? s_route[j] : -1;
            const int64_t srow = r < 0 ? -1 : (MODE == MOE_GATE_UP ? r / p.top_k : r);
            src[i] = srow < 0 ? nullptr : p.xh + srow * p.k;
        }
        int ks = 0;
        for (; ks < KS; ks++) {
            const int s = ks % MOE_STAGES;
            const uint32_t ph = (uint32_t)(ks / MOE_STAGES) & 1u;
            if (*abort_flag) break;
            if (!tc::mbar_wait(&empty[s], ph ^ 1u)) { fail(1); break; }
            const uint32_t bbase = tc::smem_u32(sB + s * moe_b_bytes(BN));
#pragma unroll
            for (int i = 0; i < RPL; i++) {
                const int j = lane + 32 * i;
                if (j >= BN) continue;
#pragma unroll
                for (int c = 0; c < 8; c++) {
                    const int64_t kk = (int64_t)ks * MOE_BK + 8 * c;
                    const bool v = src[i] != nullptr && kk < p.k;
                    cp_async16(bbase + j * 128 + ((c ^ (j & 7)) * 16), v ? (const void *)(src[i] + kk) : (const void *)p.xh,
                               v ? 16u : 0u);
                }
            }
            cp_async_commit();
            if (ks >= MOE_GATHER_LAG) {
                cp_async_wait<MOE_GATHER_LAG>();
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(&full_b[(ks - MOE_GATHER_LAG) % MOE_STAGES]);
            }
        }
        cp_async_wait<0>();
        tc::fence_proxy_async_smem();
        for (int d = ks - MOE_GATHER_LAG < 0 ? 0 : ks - MOE_GATHER_LAG; d < ks; d++) tc::mbar_arrive(&full_b[d % MOE_STAGES]);
    } else if (warp == 1) {
        // ---------------- MMA issuer (N rounded up to 16 for the last tile of an expert)
        if (lane == 0) {
            const int n_mma = ((n_eff + 15) / 16) * 16;
            const uint32_t idesc = tc::idesc_f16_f32(MOE_BM, n_mma);
            for (int ks = 0; ks < KS; ks++) {
                const int s = ks % MOE_STAGES;
                const uint32_t ph = (uint32_t)(ks / MOE_STAGES) & 1u;
                if (*abort_flag) break;
                if (!tc::mbar_wait(&full_a[s], ph) || !tc::mbar_wait(&full_b[s], ph)) { fail(2); break; }
                tc::tc_fence_after();
                const uint32_t a0 = tc::smem_u32(sA + s * MOE_A_BYTES);
                const uint32_t b0 = tc::smem_u32(sB + s * moe_b_bytes(BN));
#pragma unroll
                for (int kk = 0; kk < MOE_BK / 16; kk++)
                    tc::mma_f16(tmem, tc::sw128_desc(a0 + 32 * kk), tc::sw128_desc(b0 + 32 * kk), idesc,
                                (ks | kk) != 0 ? 1u : 0u);
                tc::mma_commit(&empty[s]);
            }
            tc::mma_commit(done);
        }
    } else {
        // ---------------- weight producers: 128 rows of expert e
        const int t = tid - 64;
        int64_t wrow_idx;
        if (MODE == MOE_GATE_UP) {
            const int64_t half = p.n / 2;  // gate rows [0, I), up rows [I, 2I)
            wrow_idx = t < 64 ? (int64_t)blockIdx.x * 64 + t : half + (int64_t)blockIdx.x * 64 + (t - 64);
        } else {
            wrow_idx = (int64_t)blockIdx.x * MOE_BM + t;
        }
        const bool live = wrow_idx < p.n;
        const uint8_t *wrow = p.w + (int64_t)e * p.expert_stride + (live ? wrow_idx : 0) * p.rb;
        KUnit<WT> u[2];
        if constexpr (WT == GGUF_Q8_0) { u[0].kblocks = p.k / 32; u[1].kblocks = p.k / 32; }
        if (live) {
            u[0].load(wrow, 0);
            if (KS > 1) u[1].load(wrow, 1);
        }
        for (int ks0 = 0; ks0 < KS; ks0 += 2) {
#pragma unroll
            for (int j = 0; j < 2; j++) {
                const int ks = ks0 + j;
                if (ks >= KS) break;
                const int s = ks % MOE_STAGES;
                const uint32_t ph = (uint32_t)(ks / MOE_STAGES) & 1u;
                uint32_t vals[32];
                if (live) u[j].unpack(ks, vals);
                else {
#pragma unroll
                    for (int i = 0; i < 32; i++) vals[i] = 0u;
                }
                if (live && ks + 2 < KS) u[j].load(wrow, ks + 2);
                if (*abort_flag) break;
                if (!tc::mbar_wait(&empty[s], ph ^ 1u)) { fail(4); break; }
                store_sw128_row(sA + s * MOE_A_BYTES, t, vals);
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(&full_a[s]);
            }
            if (*abort_flag) break;
        }

        // ---------------- epilogue
        const bool ok = tc::mbar_wait(done, 0);
        if (!ok) fail(8);
        tc::tc_fence_after();
        const bool go = ok && !*abort_flag;
        const int q = warp & 3;
        if (MODE == MOE_DOWN) {
            const int64_t orow = (int64_t)blockIdx.x * MOE_BM + 32 * q + lane;
#pragma unroll 1
            for (int c = 0; c * 32 < BN; c++) {
                uint32_t r[32];
                tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + 32 * c, r);
                tc::tmem_ld_wait();
                if (!go || orow >= p.n) continue;
#pragma unroll
                for (int jj = 0; jj < 32; jj++) {
                    const int j = 32 * c + jj;
                    if (j < n_eff) {
                        const int rr = s_route[j];
                        const int64_t tok = rr / p.top_k;
                        atomicAdd(&p.yacc[tok * p.n + orow], s_w[j] * __uint_as_float(r[jj]));
                    }
                }
            }
        } else {
            // gate rows live in TMEM lanes 0..63 (q = 0, 1), up rows in 64..127 (q = 2, 3)
            float *xbuf = reinterpret_cast<float *>(sA);  // [64][BN] up values; the operand stages are idle now
#pragma unroll 1
            for (int c = 0; c * 32 < BN; c++) {
                uint32_t r[32];
                tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + 32 * c, r);
                tc::tmem_ld_wait();
                if (q >= 2) {
#pragma unroll
                    for (int jj = 0; jj < 32; jj++)
                        if (32 * c + jj < BN) xbuf[(32 * (q - 2) + lane) * BN + 32 * c + jj] = __uint_as_float(r[jj]);
                }
                named_bar_sync(1, 128);
                if (q < 2 && go) {
                    const int il = 32 * q + lane;                       // i within the 64-row slice
                    const int64_t i = (int64_t)blockIdx.x * 64 + il;   // column of h
                    const int64_t idim = p.n / 2;
                    const int64_t hrb = idim / 32 * Q8_1_BYTES;
#pragma unroll 1
                    for (int jj = 0; jj < 32; jj++) {
                        const int j = 32 * c + jj;
                        if (j >= n_eff) break;
                        const int64_t rr = s_route[j];
                        const float gv = __uint_as_float(r[jj]);
                        const float uv = xbuf[il * BN + j];
                        const float hf = gv / (1.0f + expf(-gv)) * uv;
                        const uint16_t hb = f2bf_rn(hf);
                        const float hx = bf2f(hb);  // the activation-dtype intermediate
                        if (p.hbf) p.hbf[rr * idim + i] = hb;
                        // q8_1 of the 32 consecutive i held by this warp
                        float amax = fabsf(hx);
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                        const float d = __fdiv_rn(amax, 127.0f);
                        const int qv = d != 0.0f ? (int)roundf(__fdiv_rn(hx, d)) : 0;
                        int sum = qv;
#pragma unroll
                        for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                        const uint16_t dh = f2h_rn(d);
                        if (p.hq) {
                            uint8_t *blk = p.hq + rr * hrb + (i / 32) * Q8_1_BYTES;
                            blk[4 + lane] = (uint8_t)(int8_t)qv;
                            if (lane == 0) {
                                const uint16_t sh = f2h_rn(__fmul_rn(d, (float)sum));
                                *reinterpret_cast<uint32_t *>(blk) = (uint32_t)dh | ((uint32_t)sh << 16);
                            }
                        }
                        if (p.h16) p.h16[rr * idim + i] = f2h_rn(h2f(dh) * (float)qv);
                    }
                }
                named_bar_sync(1, 128);
            }
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, TMEM_COLS);
}

// y[t][n] (out dtype) from the fp32 accumulator
__global__ void moe_finalize_kernel(const float *__restrict__ yacc, int64_t count, void *__restrict__ y, int yt) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i < count) store_out(y, yt, i, yacc[i]);
}

// ---------------------------------------------------------------- host side

static size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

int moe_bn(int64_t routes, int64_t experts) {
    (void)routes;
    (void)experts;
    return 128;
}

// Carve the workspace (base == nullptr: only compute the size): grouping
// tables, then the fp16 activation operand, the fp32 output accumulator and
// the fp16 intermediate (each optional: 0 elements).
MoeWs moe_ws_layout(void *base, int64_t E, int64_t R, int64_t xh_elems, int64_t yacc_elems, int64_t h16_elems) {
    MoeWs w{};
    uint8_t *p = reinterpret_cast<uint8_t *>(base);
    size_t off = 0;
    auto take = [&](size_t bytes) -> void * {
        void *r = (p && bytes) ? p + off : nullptr;
        off += a256(bytes);
        return r;
    };
    const int bn = moe_bn(R, E);
    const int64_t max_tiles = (R + bn - 1) / bn + (E < R ? E : R) + 1;
    w.counts = (int32_t *)take(sizeof(int32_t) * (size_t)E);
    w.offsets = (int32_t *)take(sizeof(int32_t) * (size_t)(E + 1));
    w.pos = (int32_t *)take(sizeof(int32_t) * (size_t)R);
    w.route_list = (int32_t *)take(sizeof(int32_t) * (size_t)R);
    w.tile_expert = (int32_t *)take(sizeof(int32_t) * (size_t)max_tiles);
    w.tile_start = (int32_t *)take(sizeof(int32_t) * (size_t)max_tiles);
    w.n_tiles = (int32_t *)take(sizeof(int32_t));
    w.xh = (uint16_t *)take(sizeof(uint16_t) * (size_t)xh_elems);
    w.yacc = (float *)take(sizeof(float) * (size_t)yacc_elems);
    w.h16 = (uint16_t *)take(sizeof(uint16_t) * (size_t)h16_elems);
    w.bytes = off;
    return w;
}

cudaError_t moe_group(const int32_t *ids, const float *rw, int64_t R, int64_t E, bool skip_zero_w, int32_t *status,
                      const MoeWs &w, int bn, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(w.counts, 0, sizeof(int32_t) * (size_t)E, s);
    if (e != cudaSuccess) return e;
    const unsigned g = (unsigned)((R + 255) / 256);
    if (R > 0) moe_count_kernel<<<g, 256, 0, s>>>(ids, rw, R, E, skip_zero_w ? 1 : 0, w.counts, w.pos, status);
    moe_scan_kernel<<<1, 1024, 0, s>>>(w.counts, E, bn, w.offsets, w.tile_expert, w.tile_start, w.n_tiles);
    if (R > 0) moe_scatter_kernel<<<g, 256, 0, s>>>(ids, w.pos, R, w.offsets, w.route_list);
    return cudaGetLastError();
}

template <int WT, int BN, int MODE>
static cudaError_t launch_moe_t(const MoeParams &p, int64_t max_tiles, cudaStream_t s) {
    auto kern = moe_mmq_kernel<WT, BN, MODE>;
    constexpr int smem = moe_smem_bytes(BN);
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    const int64_t gx = MODE == MOE_GATE_UP ? p.n / 2 / 64 : (p.n + MOE_BM - 1) / MOE_BM;
    dim3 grid((unsigned)gx, (unsigned)max_tiles);
    kern<<<grid, MOE_THREADS, smem, s>>>(p);
    return cudaGetLastError();
}

template <int MODE>
static cudaError_t launch_moe_mode(int wt, const MoeParams &p, int64_t max_tiles, cudaStream_t s) {
    switch (wt) {
    case GGUF_Q4_K: return launch_moe_t<GGUF_Q4_K, 128, MODE>(p, max_tiles, s);
    case GGUF_Q6_K: return launch_moe_t<GGUF_Q6_K, 128, MODE>(p, max_tiles, s);
    case GGUF_Q8_0: return launch_moe_t<GGUF_Q8_0, 128, MODE>(p, max_tiles, s);
    default: return cudaErrorInvalidValue;
    }
}

// gate_up: h rows per route from token rows xh [T][k]
cudaError_t launch_moe_gate_up(const uint8_t *w, int wt, int64_t expert_stride, int64_t n, int64_t k,
                               const uint16_t *xh, int64_t top_k, int64_t R, int64_t E, const MoeWs &ws,
                               uint8_t *hq, uint16_t *hbf, uint16_t *h16, cudaStream_t s) {
    const int bn = moe_bn(R, E);
    MoeParams p{};
    p.w = w; p.expert_stride = expert_stride; p.rb = k / block_elems(wt) * block_bytes(wt); p.n = n; p.k = k;
    p.xh = xh; p.top_k = top_k;
    p.route_list = ws.route_list; p.offsets = ws.offsets; p.counts = ws.counts;
    p.tile_expert = ws.tile_expert; p.tile_start = ws.tile_start; p.n_tiles = ws.n_tiles;
    p.hq = hq; p.hbf = hbf; p.h16 = h16;
    const int64_t max_tiles = (R + bn - 1) / bn + (E < R ? E : R) + 1;
    if (R == 0) return cudaSuccess;
    return launch_moe_mode<MOE_GATE_UP>(wt, p, max_tiles, s);
}

// down: y_acc[T][n] += route_w * (W[e] . xh[route])
cudaError_t launch_moe_down(const uint8_t *w, int wt, int64_t expert_stride, int64_t n, int64_t k,
                            const uint16_t *xh, int64_t top_k, int64_t R, int64_t E, const float *route_w,
                            const MoeWs &ws, float *yacc, cudaStream_t s) {
    const int bn = moe_bn(R, E);
    MoeParams p{};
    p.w = w; p.expert_stride = expert_stride; p.rb = k / block_elems(wt) * block_bytes(wt); p.n = n; p.k = k;
    p.xh = xh; p.top_k = top_k;
    p.route_list = ws.route_list; p.offsets = ws.offsets; p.counts = ws.counts;
    p.tile_expert = ws.tile_expert; p.tile_start = ws.tile_start; p.n_tiles = ws.n_tiles;
    p.route_w = route_w; p.yacc = yacc;
    const int64_t max_tiles = (R + bn - 1) / bn + (E < R ? E : R) + 1;
    if (R == 0) return cudaSuccess;
    return launch_moe_mode<MOE_DOWN>(wt, p, max_tiles, s);
}

cudaError_t launch_moe_finalize(const float *yacc, int64_t count, void *y, int yt, cudaStream_t s) {
    if (count == 0) return cudaSuccess;
    moe_finalize_kernel<<<(unsigned)((count + 255) / 256), 256, 0, s>>>(yacc, count, y, yt);
    return cudaGetLastError();
}

}  // namespace gg
