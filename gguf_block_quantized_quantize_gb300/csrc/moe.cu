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
// GEMM tile: 128 weight rows x BN routes x 64 K per stage, the same fp16
// tcgen05 engine as the dense MMQ.  The activation rows of a tile are loaded
// as one 2-D box per K-step; the last tile of an expert issues the MMA with N
// rounded up to 16 only.
// The activation operand is written in grouped route order (the conversion
// quantizes each token row once and writes it to the grouped row of each of
// its active routes), so an expert's routes are consecutive rows and a tile
// loads them with plain 2-D bulk tensor copies instead of per-row gathers.
//   gate_up : the A tile holds 64 gate rows i and the 64 matching up rows I+i,
//             so the epilogue has g and u of the same (route, i): it computes
//             h = silu(g) * u in fp32, rounds it to bf16 (the activation dtype),
//             quantizes each 32 consecutive i (one warp) to a q8_1 block, and
//             writes q8_1 / bf16 (per route) or fp16 (d16*q, the operand of the
//             down GEMM, in grouped order).
//   down    : z[route][n] = W_down[e] . h_route (fp32, plain stores); a last
//             pass sums each token's routes in slot order, y[t] = sum_k w_k z,
//             so the result is deterministic and needs no atomics.
#include <mutex>

#include "tcgemm.cuh"

namespace gg {

constexpr int MOE_BN = 128;  // routes per work tile

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

// The same counts with a per-CTA histogram in shared memory (E <= 8192): each
// CTA takes MOE_COUNT_CHUNK consecutive routes, gives each active one its
// place among the CTA's routes of its expert, then adds the CTA's count of
// every expert to counts[] once (one global atomic per expert and CTA instead
// of one per route) and shifts its routes' places by the returned base.
constexpr int MOE_COUNT_CHUNK = 4096;
__global__ void __launch_bounds__(256) moe_count_smem_kernel(const int32_t *__restrict__ ids,
                                                             const float *__restrict__ rw, int64_t R, int64_t E,
                                                             int skip_zero_w, int32_t *__restrict__ counts,
                                                             int32_t *__restrict__ pos,
                                                             int32_t *__restrict__ dev_status) {
    extern __shared__ int32_t hist[];   // [E] local counts, then the global bases
    for (int64_t e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
    __syncthreads();
    const int64_t r0 = (int64_t)blockIdx.x * MOE_COUNT_CHUNK;
    const int64_t r1 = r0 + MOE_COUNT_CHUNK < R ? r0 + MOE_COUNT_CHUNK : R;
    int bad = 0;
    for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
        const int32_t e = ids[r];
        const bool ok = e >= 0 && e < E && !(skip_zero_w && rw != nullptr && rw[r] == 0.0f);
        bad += e >= E;
        pos[r] = ok ? atomicAdd(&hist[e], 1) : -1;
    }
    if (bad && dev_status != nullptr) atomicAdd(dev_status, bad);
    __syncthreads();
    for (int64_t e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t c = hist[e];
        hist[e] = c ? atomicAdd(&counts[e], c) : 0;
    }
    __syncthreads();
    for (int64_t r = r0 + threadIdx.x; r < r1; r += blockDim.x) {
        const int32_t p = pos[r];
        if (p >= 0) pos[r] = p + hist[ids[r]];
    }
}

// the route marks of the route-batched path: pos[r] = r for an active route,
// -1 for a skipped one (same rules as moe_count_kernel; no grouping needed)
__global__ void moe_mark_kernel(const int32_t *__restrict__ ids, const float *__restrict__ rw, int64_t R, int64_t E,
                                int skip_zero_w, int32_t *__restrict__ pos, int32_t *__restrict__ dev_status) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= R) return;
    const int32_t e = ids[r];
    const bool ok = e >= 0 && e < E && !(skip_zero_w && rw != nullptr && rw[r] == 0.0f);
    if (e >= E && dev_status != nullptr) atomicAdd(dev_status, 1);
    pos[r] = ok ? (int32_t)r : -1;
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

// y[t][c] = sum over the token's route slots k (in order) of w_k * z(t*top_k + k, c);
// routes that were not grouped (inactive id, or weight 0) have pos = -1 and no z row.
// z is [R][n] in route order, or, with offsets, the grouped GEMM's layout:
// route r at its grouped position g = offsets[ids[r]] + pos[r], column c at
// ((c / 128) * R + g) * 128 + c % 128.  V consecutive columns per thread
// (V = 4 when n % 4 == 0: 16-byte loads)
template <int V>
__global__ void moe_finalize_kernel(const float *__restrict__ z, const int32_t *__restrict__ pos,
                                    const int32_t *__restrict__ ids, const int32_t *__restrict__ offsets,
                                    const float *__restrict__ route_w, int64_t T, int64_t top_k, int64_t n,
                                    void *__restrict__ y, int yt) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // z comes from the previous kernel
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * V;
    if (i >= T * n) return;
    const int64_t t = i / n, c = i - t * n;
    float acc[V];
#pragma unroll
    for (int v = 0; v < V; v++) acc[v] = 0.0f;
    // routes in groups of 8: every index and z load of a group is issued before
    // the group's products are added, in slot order
    constexpr int KG = 8;
    for (int64_t k0 = 0; k0 < top_k; k0 += KG) {
        int64_t zi[KG];
        float wk[KG];
#pragma unroll
        for (int j = 0; j < KG; j++) {
            const int64_t r = t * top_k + k0 + j;
            const int32_t pr = k0 + j < top_k ? pos[r] : -1;
            wk[j] = pr < 0 ? 0.0f : (route_w ? route_w[r] : 1.0f);
            // grouped rows are stored in 128-column blocks of R rows
            zi[j] = pr < 0 ? -1
                           : offsets ? ((((c >> 7) * T * top_k) + offsets[ids[r]] + pr) << 7) + (c & 127) : r * n + c;
        }
        if (V == 4) {
            float4 zv[KG];
#pragma unroll
            for (int j = 0; j < KG; j++)
                zv[j] = zi[j] < 0 ? make_float4(0.0f, 0.0f, 0.0f, 0.0f) : *reinterpret_cast<const float4 *>(z + zi[j]);
#pragma unroll
            for (int j = 0; j < KG; j++) {
                if (zi[j] < 0) continue;   // a skipped route adds nothing (not even a zero)
                acc[0] = fmaf(wk[j], zv[j].x, acc[0]);
                acc[1] = fmaf(wk[j], zv[j].y, acc[1]);
                acc[2] = fmaf(wk[j], zv[j].z, acc[2]);
                acc[3] = fmaf(wk[j], zv[j].w, acc[3]);
            }
        } else {
#pragma unroll
            for (int j = 0; j < KG; j++) {
                if (zi[j] < 0) continue;
                const int64_t r = t * top_k + k0 + j;
#pragma unroll
                for (int v = 0; v < V; v++) {
                    const int64_t cv = c + v;
                    const int64_t zv = offsets ? ((((cv >> 7) * T * top_k) + offsets[ids[r]] + pos[r]) << 7) + (cv & 127)
                                               : r * n + cv;
                    acc[v] = fmaf(wk[j], z[zv], acc[v]);
                }
            }
        }
    }
#pragma unroll
    for (int v = 0; v < V; v++) store_out(y, yt, i + v, acc[v]);
}

// SwiGLU of the route-batched gate_up: h = silu(g) * u in fp32 (IEEE exp and
// division), rounded to bf16, the activation dtype
__global__ void moe_swiglu_kernel(const float *__restrict__ z, const int32_t *__restrict__ pos, int64_t R, int64_t I,
                                  uint16_t *__restrict__ h) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // z comes from the previous kernel
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= R * I) return;
    const int64_t r = i / I, j = i - r * I;
    uint16_t bits = 0;
    if (pos[r] >= 0) {
        const float g = z[r * 2 * I + j], u = z[r * 2 * I + I + j];
        bits = f2bf_rn(g / (1.0f + expf(-g)) * u);
    }
    h[i] = bits;
}

// The same SwiGLU and the q8_1 quantization of h in one pass (the down
// product's input): four threads per 32-value block, each rounding 8 values
// of h to bf16 and quantizing them by the rule of the q8_1 quantize kernel
// (d = amax / 127, q = roundf(h / d), s = fp16(d * sum q)), so the blocks are
// the bits that quantizing the bf16 rows gives.  Skipped routes get zero
// blocks, as their zero rows would.
__global__ void __launch_bounds__(256) moe_swiglu_q8_1_kernel(const float *__restrict__ z,
                                                              const int32_t *__restrict__ pos, int64_t R, int64_t I,
                                                              uint8_t *__restrict__ hq) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // z comes from the previous kernel
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t nb = I / 32;
    const int64_t gidx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t blk = gidx >> 2;
    const int j = (int)(gidx & 3);
    const bool in = blk < R * nb;
    const int64_t r = in ? blk / nb : 0, b = in ? blk - r * nb : 0;
    const bool on = in && pos[r] >= 0;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; i++) {
        float hx = 0.0f;
        if (on) {
            const int64_t c = b * 32 + 8 * j + i;
            const float g = z[r * 2 * I + c], u = z[r * 2 * I + I + c];
            hx = bf2f(f2bf_rn(g / (1.0f + expf(-g)) * u));
        }
        v[i] = hx;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);
    int q[8], sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        q[i] = (d != 0.0f) ? (int)roundf(__fdiv_rn(v[i], d)) : 0;
        sum += q[i];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    if (!in) return;
    uint8_t *o = hq + blk * Q8_1_BYTES;
    const uint32_t w0 = (q[0] & 0xff) | ((q[1] & 0xff) << 8) | ((q[2] & 0xff) << 16) | ((uint32_t)(q[3] & 0xff) << 24);
    const uint32_t w1 = (q[4] & 0xff) | ((q[5] & 0xff) << 8) | ((q[6] & 0xff) << 16) | ((uint32_t)(q[7] & 0xff) << 24);
    reinterpret_cast<uint32_t *>(o + 4 + 8 * j)[0] = w0;
    reinterpret_cast<uint32_t *>(o + 4 + 8 * j)[1] = w1;
    if (j == 0) {
        const uint16_t dh = f2h_rn(d), sh = f2h_rn(__fmul_rn(d, (float)sum));
        *reinterpret_cast<uint32_t *>(o) = (uint32_t)dh | ((uint32_t)sh << 16);
    }
}

// ---------------------------------------------------------------- host side

// a 1-D launch that may start while the previous kernel of the stream
// finishes (the kernel waits on griddepcontrol before reading its inputs)
template <typename... KArgs, typename... Args>
static cudaError_t launch_pdl(void (*kern)(KArgs...), int64_t blocks, unsigned threads, cudaStream_t s, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

static size_t a256(size_t v) { return (v + 255) & ~size_t(255); }

int moe_bn(int64_t routes, int64_t experts) {
    (void)routes;
    (void)experts;
    return MOE_BN;
}

// Carve the workspace (base == nullptr: only compute the size): grouping
// tables, the fp16 activation operand (hi and lo parts), the fp32 per-route
// outputs of the down GEMM and the fp16 intermediate (each optional: 0 elements).
MoeWs moe_ws_layout(void *base, int64_t E, int64_t R, int64_t xh_elems, int64_t z_elems, int64_t h16_elems,
                    bool with_lo, int64_t vec_n2) {
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
    w.xl = (uint16_t *)take(sizeof(uint16_t) * (size_t)xh_elems);  // low parts: the gate_up is always precise
    w.z = (float *)take(sizeof(float) * (size_t)z_elems);
    w.h16 = (uint16_t *)take(sizeof(uint16_t) * (size_t)h16_elems);
    w.h16lo = (uint16_t *)take(sizeof(uint16_t) * (size_t)(with_lo ? h16_elems : 0));
    w.zv = (float *)take(sizeof(float) * (size_t)(R * vec_n2));
    w.hb = (uint16_t *)take(sizeof(uint16_t) * (size_t)(R * vec_n2 / 2));
    w.hqv = (uint8_t *)take((size_t)(R * (vec_n2 / 2 / 32) * Q8_1_BYTES));
    w.bytes = off;
    return w;
}

cudaError_t moe_group(const int32_t *ids, const float *rw, int64_t R, int64_t E, bool skip_zero_w, int32_t *status,
                      const MoeWs &w, int bn, cudaStream_t s) {
    cudaError_t e = cudaMemsetAsync(w.counts, 0, sizeof(int32_t) * (size_t)E, s);
    if (e != cudaSuccess) return e;
    const unsigned g = (unsigned)((R + 255) / 256);
    if (R > 0 && E <= 8192)
        moe_count_smem_kernel<<<(unsigned)((R + MOE_COUNT_CHUNK - 1) / MOE_COUNT_CHUNK), 256, (size_t)E * 4, s>>>(
            ids, rw, R, E, skip_zero_w ? 1 : 0, w.counts, w.pos, status);
    else if (R > 0)
        moe_count_kernel<<<g, 256, 0, s>>>(ids, rw, R, E, skip_zero_w ? 1 : 0, w.counts, w.pos, status);
    moe_scan_kernel<<<1, 1024, 0, s>>>(w.counts, E, bn, w.offsets, w.tile_expert, w.tile_start, w.n_tiles);
    if (R > 0) moe_scatter_kernel<<<g, 256, 0, s>>>(ids, w.pos, R, w.offsets, w.route_list);
    return cudaGetLastError();
}

// rows: operand rows in grouped route order (R), each p.kx fp16; a tile
// reads 64 values of its 128 consecutive rows per K-step
template <int WT, int MODE, bool PRECISE>
static cudaError_t launch_moe_wt(TgParams p, int64_t rows, int64_t n_experts, cudaStream_t s) {
    CUtensorMap mh{}, ml{}, mw{};
    cudaError_t e = tg_make_map(&mh, p.xh, rows, p.kx, MOE_BN);
    if (e == cudaSuccess && PRECISE) e = tg_make_map(&ml, p.xl, rows, p.kx, MOE_BN);
    if (e != cudaSuccess) return e;
    if (option_mmq_stage())   // gate_up buffers: 64 gate rows and the 64 matching up rows
        tg_plan_staging(p, &mw, WT, p.w, p.n, n_experts, p.expert_stride, p.k, MODE == TG_MOE_GATE_UP ? 64 : TG_BM,
                        tg_base_bytes<WT, MOE_BN, PRECISE, MODE>());
    const int grid = device_info().sm_count;  // persistent; CTAs beyond the device-side tile count exit
    return tg_launch<WT, MOE_BN, PRECISE, MODE, GGUF_F32>(mh, ml, mw, mh, p, grid, s);
}

template <int MODE, bool PRECISE>
static cudaError_t launch_moe_mode(int wt, const TgParams &p, int64_t rows, int64_t n_experts, cudaStream_t s) {
    switch (wt) {
    case GGUF_Q4_K: return launch_moe_wt<GGUF_Q4_K, MODE, PRECISE>(p, rows, n_experts, s);
    case GGUF_Q6_K: return launch_moe_wt<GGUF_Q6_K, MODE, PRECISE>(p, rows, n_experts, s);
    case GGUF_Q8_0: return launch_moe_wt<GGUF_Q8_0, MODE, PRECISE>(p, rows, n_experts, s);
    case GGUF_Q4_0: return launch_moe_wt<GGUF_Q4_0, MODE, PRECISE>(p, rows, n_experts, s);
    case GGUF_Q5_K: return launch_moe_wt<GGUF_Q5_K, MODE, PRECISE>(p, rows, n_experts, s);
    case GGUF_MXFP4: return launch_moe_wt<GGUF_MXFP4, MODE, PRECISE>(p, rows, n_experts, s);
    default: return cudaErrorInvalidValue;
    }
}

static TgParams moe_params(const uint8_t *w, int wt, int64_t expert_stride, int64_t n, int64_t k, const uint16_t *xh,
                           const uint16_t *xl, int64_t top_k, const MoeWs &ws) {
    TgParams p{};
    p.w = w;
    p.expert_stride = expert_stride;
    p.rb = k / block_elems(wt) * block_bytes(wt);
    p.n = n;
    p.k = k;
    p.kx = op_pitch(wt, k);
    p.xh = xh;
    p.xl = xl;
    p.top_k = top_k;
    p.route_list = ws.route_list;
    p.offsets = ws.offsets;
    p.counts = ws.counts;
    p.tile_expert = ws.tile_expert;
    p.tile_start = ws.tile_start;
    p.n_tiles = ws.n_tiles;
    return p;
}

// gate_up (+ SwiGLU + q8_1); xh / xl: the operand rows in grouped route order
// [R][kx]; with xl (the low parts) the product runs in the precise (hi + lo)
// mode, else on one fp16 operand per side
cudaError_t launch_moe_gate_up(const uint8_t *w, int wt, int64_t expert_stride, int64_t n, int64_t k,
                               const uint16_t *xh, const uint16_t *xl, int64_t top_k, int64_t R, int64_t E,
                               const MoeWs &ws, uint8_t *hq, uint16_t *hbf, uint16_t *h16, uint16_t *h16lo,
                               int64_t hpitch, bool h16_grouped, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    TgParams p = moe_params(w, wt, expert_stride, n, k, xh, xl, top_k, ws);
    p.h16_grouped = h16_grouped ? 1 : 0;
    p.hpitch = hpitch < n / 2 ? n / 2 : hpitch;
    p.tiles_x = (int)(n / 2 / 64);
    p.hq = hq;
    p.hbf = hbf;
    p.h16 = h16;
    p.h16lo = h16lo;
    p.m = R / top_k;
    return xl ? launch_moe_mode<TG_MOE_GATE_UP, true>(wt, p, R, E, s)
              : launch_moe_mode<TG_MOE_GATE_UP, false>(wt, p, R, E, s);
}

// down: z[R][n] = W[e] . x[route] for every grouped route, or, with ysum,
// ysum[t][n] += route_w[r] * (W[e] . x[route]) into zeroed token rows (bulk
// reduce-adds of the staged rows when n % 4 == 0, else fp32 atomics); xh / xl:
// the operand rows in grouped route order [R][kx] (xl only in the precise mode)
cudaError_t launch_moe_down(const uint8_t *w, int wt, int64_t expert_stride, int64_t n, int64_t k,
                            const uint16_t *xh, const uint16_t *xl, int64_t top_k, int64_t R, int64_t E,
                            const MoeWs &ws, float *z, bool precise, cudaStream_t s, float *ysum,
                            const float *route_w) {
    if (R == 0) return cudaSuccess;
    TgParams p = moe_params(w, wt, expert_stride, n, k, xh, xl, top_k, ws);
    p.tiles_x = (int)((n + TG_BM - 1) / TG_BM);
    p.yacc = z;
    p.zrows = R;
    p.ysum = ysum;
    p.ysum_bulk = ysum && n % 4 == 0 && (reinterpret_cast<uintptr_t>(ysum) & 15) == 0;
    p.route_w = route_w;
    p.m = R / top_k;
    return precise ? launch_moe_mode<TG_MOE_DOWN, true>(wt, p, R, E, s)
                   : launch_moe_mode<TG_MOE_DOWN, false>(wt, p, R, E, s);
}

// y[r][c] = z(r, c) for an active route, 0 for a skipped one (out dtype); the
// layouts of z as in the finalize
__global__ void moe_plain_store_kernel(const float *__restrict__ z, const int32_t *__restrict__ pos,
                                       const int32_t *__restrict__ ids, const int32_t *__restrict__ offsets,
                                       int64_t R, int64_t n, void *__restrict__ y, int yt) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // z comes from the previous kernel
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= R * n) return;
    const int64_t r = i / n, c = i - r * n;
    const int32_t pr = pos[r];
    const int64_t zi = offsets ? ((((c >> 7) * R) + (pr >= 0 ? offsets[ids[r]] + pr : 0)) << 7) + (c & 127) : i;
    store_out(y, yt, i, pr >= 0 ? z[zi] : 0.0f);
}

cudaError_t launch_moe_plain_store(const float *z, const int32_t *pos, const int32_t *ids, const int32_t *offsets,
                                   int64_t R, int64_t n, void *y, int yt, cudaStream_t s) {
    const int64_t count = R * n;
    if (count == 0) return cudaSuccess;
    return launch_pdl(moe_plain_store_kernel, (count + 255) / 256, 256, s, z, pos, ids, offsets, R, n, y, yt);
}

// y[T][n] = the route-weighted sum of each token's z rows (out dtype)
cudaError_t launch_moe_finalize(const float *z, const int32_t *pos, const int32_t *ids, const int32_t *offsets,
                                const float *route_w, int64_t T, int64_t top_k, int64_t n, void *y, int yt,
                                cudaStream_t s) {
    const int64_t count = T * n;
    if (count == 0) return cudaSuccess;
    if (n % 4 == 0)   // z rows are 16-byte aligned (workspace base 256-aligned, n % 4 == 0)
        return launch_pdl(moe_finalize_kernel<4>, (count / 4 + 255) / 256, 256, s, z, pos, ids, offsets, route_w, T,
                          top_k, n, y, yt);
    return launch_pdl(moe_finalize_kernel<1>, (count + 255) / 256, 256, s, z, pos, ids, offsets, route_w, T, top_k, n,
                      y, yt);
}

cudaError_t launch_moe_swiglu_q8_1(const float *z, const int32_t *pos, int64_t R, int64_t I, uint8_t *hq,
                                  cudaStream_t s) {
    const int64_t threads = R * (I / 32) * 4;
    if (threads == 0) return cudaSuccess;
    return launch_pdl(moe_swiglu_q8_1_kernel, (threads + 255) / 256, 256, s, z, pos, R, I, hq);
}

cudaError_t launch_moe_swiglu(const float *z, const int32_t *pos, int64_t R, int64_t I, uint16_t *h, cudaStream_t s) {
    const int64_t count = R * I;
    if (count == 0) return cudaSuccess;
    return launch_pdl(moe_swiglu_kernel, (count + 255) / 256, 256, s, z, pos, R, I, h);
}

cudaError_t moe_mark(const int32_t *ids, const float *rw, int64_t R, int64_t E, bool skip_zero_w, int32_t *status,
                     int32_t *pos, cudaStream_t s) {
    if (R == 0) return cudaSuccess;
    return launch_pdl(moe_mark_kernel, (R + 255) / 256, 256, s, ids, rw, R, E, skip_zero_w ? 1 : 0, pos, status);
}

}  // namespace gg
