// MMVQ: quantized weight x q8_1 activation product for small token counts
// (decode).  y[m][n] = sum over the row's sub-blocks of an exact int32 block
// dot product combined with the fp32 block scales:
//   Q8_0: d_w * d_a * S
//   Q4_K: d * s_j * d_a * S_j - dmin * m_j * s_a
//   Q6_K: d * sc_j * d_a * S_j
// (FreeToken PR #690 "serve GGUF checkpoints on vendored ggml-cuda kernels",
// section "Vendored ggml": q8_1 activations, fp32 accumulation, results in the
// activation dtype; MMVQ serves the small batches, section "Changes").
//
// GB300 design.  The kernel is bound by the HBM read of the packed weights
// (transformers PR #45977 "GgufLinear ...", section "What made it fast": a
// bandwidth-bound decode), so every weight byte is read exactly once, with
// coalesced loads, and all compute hides under those loads:
//   * K is split across the threads of a CTA: thread t owns the 32-value
//     "pieces" t, t + blockDim, ... of every row.  Its q8_1 activation quants
//     for those pieces (all m rows) are loaded once into registers and reused
//     for every weight row the CTA visits, so activations cost no bandwidth in
//     the row loop.
//   * A persistent grid (a few CTAs per SM) walks the rows R at a time; the R
//     rows' loads are issued together to keep enough bytes in flight.
//   * Per-piece int32 sums use dp4a; partial sums of the R x M outputs are
//     reduced with a butterfly (one shuffle per value and level) and then
//     across warps through shared memory.
// Piece p of a row (32 values):
//   Q8_0: block p.
//   Q4_K: super-block p/8, 16 quant bytes at chunk c = (p%8)/2, half h = p%2:
//         values [64c+16h, +16) (low nibbles, sub-block 2c) and
//         [64c+32+16h, +16) (high nibbles, sub-block 2c+1).
//   Q6_K: super-block p/8, half h = (p%8)/4, l0 = 8*(p%4): the runs
//         [128h + 32g + l0, +8) for g = 0..3.
#pragma once

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gg {

template <int M>
struct ActPiece {
    int q[M][8];      // activation quants of the piece, 4 per word, in piece order
    float f[M][4];    // Q8_0: d_a | Q4_K: d_a0, d_a1, s_a0, s_a1 | Q6_K: d_a of runs 0..3
    int sum[M][4];    // Q6_K: sum of the 8 activation quants of each run
};

// q8_1 block fields
__device__ __forceinline__ void q81_load(const uint8_t *blk, float &d, float &s) {
    const uint32_t ds = ld_u32(blk);
    d = h2f(ds & 0xffff);
    s = h2f(ds >> 16);
}

__device__ __forceinline__ int bsum4(int w) {
    return (int)(int8_t)(w) + (int)(int8_t)(w >> 8) + (int)(int8_t)(w >> 16) + (int)(int8_t)(w >> 24);
}

template <int WT, int M>
__device__ __forceinline__ void load_act(ActPiece<M> &a, const uint8_t *xq, int64_t xrb, int m_act, int64_t p,
                                         bool valid) {
#pragma unroll
    for (int mm = 0; mm < M; mm++) {
#pragma unroll
        for (int i = 0; i < 8; i++) a.q[mm][i] = 0;
#pragma unroll
        for (int i = 0; i < 4; i++) { a.f[mm][i] = 0.0f; a.sum[mm][i] = 0; }
        if (!valid || mm >= m_act) continue;
        const uint8_t *row = xq + mm * xrb;
        if (WT == GGUF_Q8_0) {
            const uint8_t *blk = row + p * Q8_1_BYTES;
            float d, s;
            q81_load(blk, d, s);
            a.f[mm][0] = d;
#pragma unroll
            for (int i = 0; i < 8; i++) a.q[mm][i] = (int)ld_u32(blk + 4 + 4 * i);
        } else if (WT == GGUF_Q4_K) {
            const int64_t sb = p >> 3;
            const int pp = (int)(p & 7), c = pp >> 1, h = pp & 1;
            const uint8_t *b0 = row + (sb * 8 + 2 * c) * Q8_1_BYTES;
            const uint8_t *b1 = b0 + Q8_1_BYTES;
            q81_load(b0, a.f[mm][0], a.f[mm][2]);
            q81_load(b1, a.f[mm][1], a.f[mm][3]);
#pragma unroll
            for (int i = 0; i < 4; i++) {
                a.q[mm][i] = (int)ld_u32(b0 + 4 + 16 * h + 4 * i);
                a.q[mm][4 + i] = (int)ld_u32(b1 + 4 + 16 * h + 4 * i);
            }
        } else {  // Q6_K
            const int64_t sb = p >> 3;
            const int pp = (int)(p & 7), h = pp >> 2, l0 = 8 * (pp & 3);
#pragma unroll
            for (int g = 0; g < 4; g++) {
                const uint8_t *b = row + (sb * 8 + 4 * h + g) * Q8_1_BYTES;
                float d, s;
                q81_load(b, d, s);
                a.f[mm][g] = d;
                a.q[mm][2 * g] = (int)ld_u32(b + 4 + l0);
                a.q[mm][2 * g + 1] = (int)ld_u32(b + 8 + l0);
                a.sum[mm][g] = bsum4(a.q[mm][2 * g]) + bsum4(a.q[mm][2 * g + 1]);
            }
        }
    }
}

// raw weight bytes of one piece, loaded before any arithmetic so that the
// loads of several rows are in flight together
template <int WT>
struct WPiece {
    uint32_t a[8];
    uint32_t b[4];
};

template <int WT>
__device__ __forceinline__ void load_w(WPiece<WT> &wp, const uint8_t *row, int64_t p) {
    if (WT == GGUF_Q8_0) {
        // d at +0 (2-aligned), quants at +2; blocks are 34 bytes, so 2-aligned
        const uint8_t *blk = row + p * Q8_0_BYTES;
        const uintptr_t qa = reinterpret_cast<uintptr_t>(blk + 2);
        if (qa & 2) {
            // quants start 2 bytes into an aligned word: words cover [blk, blk+32),
            // the last two quant bytes come from a 16-bit load (no read past the block)
            const uint8_t *base = blk;
#pragma unroll
            for (int i = 0; i < 8; i++) wp.a[i] = ld_u32(base + 4 * i);
            wp.b[0] = ld_u16(blk + 32);
            wp.b[1] = 1;  // misaligned marker
        } else {
            wp.b[0] = ld_u16(blk);  // d
#pragma unroll
            for (int i = 0; i < 8; i++) wp.a[i] = ld_u32(blk + 2 + 4 * i);
            wp.b[1] = 0;
        }
    } else if (WT == GGUF_Q4_K) {
        const int64_t sb = p >> 3;
        const int pp = (int)(p & 7), c = pp >> 1, h = pp & 1;
        const uint8_t *blk = row + sb * Q4_K_BYTES;
        const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
        const uint4 qv = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c + 16 * h);
        wp.a[0] = qv.x; wp.a[1] = qv.y; wp.a[2] = qv.z; wp.a[3] = qv.w;
        wp.b[0] = hdr.x; wp.b[1] = hdr.y; wp.b[2] = hdr.z; wp.b[3] = hdr.w;
    } else {  // Q6_K
        const int64_t sb = p >> 3;
        const int pp = (int)(p & 7), h = pp >> 2, l0 = 8 * (pp & 3);
        const uint8_t *blk = row + sb * Q6_K_BYTES;
        ld8_a2(blk + 64 * h + l0, wp.a[0], wp.a[1]);
        ld8_a2(blk + 64 * h + 32 + l0, wp.a[2], wp.a[3]);
        ld8_a2(blk + 128 + 32 * h + l0, wp.a[4], wp.a[5]);
        ld8_a2(blk + 192 + 8 * h, wp.b[0], wp.b[1]);
        wp.b[2] = ld_u16(blk + 208);
        wp.b[3] = (uint32_t)l0;
    }
}

template <int WT, int M>
__device__ __forceinline__ void dot_piece(const WPiece<WT> &wp, const ActPiece<M> &a, int64_t p, float acc[M]) {
    if (WT == GGUF_Q8_0) {
        uint32_t q[8];
        float d;
        if (wp.b[1]) {
            d = h2f(wp.a[0] & 0xffff);
#pragma unroll
            for (int i = 0; i < 7; i++) q[i] = __funnelshift_r(wp.a[i], wp.a[i + 1], 16);
            q[7] = __funnelshift_r(wp.a[7], wp.b[0], 16);
        } else {
            d = h2f(wp.b[0]);
#pragma unroll
            for (int i = 0; i < 8; i++) q[i] = wp.a[i];
        }
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
            int S = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) S = dp4a_ss((int)q[i], a.q[mm][i], S);
            acc[mm] = fmaf(d * a.f[mm][0], (float)S, acc[mm]);
        }
    } else if (WT == GGUF_Q4_K) {
        const int pp = (int)(p & 7), c = pp >> 1, h = pp & 1;
        const uint32_t sc[3] = {wp.b[1], wp.b[2], wp.b[3]};
        const float d = h2f(wp.b[0] & 0xffff), dmin = h2f(wp.b[0] >> 16);
        int s0, m0, s1, m1;
        q4k_scale_min(sc, 2 * c, s0, m0);
        q4k_scale_min(sc, 2 * c + 1, s1, m1);
        const float ds0 = d * (float)s0, ds1 = d * (float)s1;
        // the min term of a 32-value sub-block is counted once, by its h == 0 piece
        const float dm = h == 0 ? dmin : 0.0f;
        const float fm0 = (float)m0, fm1 = (float)m1;
        uint32_t lo[4], hi[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            lo[i] = wp.a[i] & 0x0F0F0F0Fu;
            hi[i] = (wp.a[i] >> 4) & 0x0F0F0F0Fu;
        }
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
            int S0 = 0, S1 = 0;
#pragma unroll
            for (int i = 0; i < 4; i++) {
                S0 = dp4a_us(lo[i], a.q[mm][i], S0);
                S1 = dp4a_us(hi[i], a.q[mm][4 + i], S1);
            }
            float v = ds0 * (a.f[mm][0] * (float)S0);
            v = fmaf(ds1, a.f[mm][1] * (float)S1, v);
            v = fmaf(-dm, fmaf(fm0, a.f[mm][2], fm1 * a.f[mm][3]), v);
            acc[mm] += v;
        }
    } else {  // Q6_K
        const int l0 = (int)wp.b[3];
        const float d = h2f(wp.b[2] & 0xffff);
        float dsc[4];
#pragma unroll
        for (int g = 0; g < 4; g++) {
            const int si = (l0 >> 4) + 2 * g;
            const int sc = (int)(int8_t)((wp.b[si >> 2] >> (8 * (si & 3))) & 0xff);
            dsc[g] = d * (float)sc;
        }
        uint32_t q[4][2];
#pragma unroll
        for (int i = 0; i < 2; i++) {
            const uint32_t A = wp.a[i], B = wp.a[2 + i], H = wp.a[4 + i];
            q[0][i] = (A & 0x0F0F0F0Fu) | ((H << 4) & 0x30303030u);
            q[1][i] = (B & 0x0F0F0F0Fu) | ((H << 2) & 0x30303030u);
            q[2][i] = ((A >> 4) & 0x0F0F0F0Fu) | (H & 0x30303030u);
            q[3][i] = ((B >> 4) & 0x0F0F0F0Fu) | ((H >> 2) & 0x30303030u);
        }
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
            float v = 0.0f;
#pragma unroll
            for (int g = 0; g < 4; g++) {
                int S = dp4a_us(q[g][0], a.q[mm][2 * g], 0);
                S = dp4a_us(q[g][1], a.q[mm][2 * g + 1], S);
                S -= 32 * a.sum[mm][g];
                v = fmaf(dsc[g], a.f[mm][g] * (float)S, v);
            }
            acc[mm] += v;
        }
    }
}

// Butterfly reduction of V values across the 32 lanes of a warp; afterwards
// lane l holds the warp total of value index l >> (5 - log2 V).
template <int V>
__device__ __forceinline__ float butterfly(float (&v)[V], int lane) {
    constexpr int LOG = V == 1 ? 0 : V == 2 ? 1 : V == 4 ? 2 : V == 8 ? 3 : V == 16 ? 4 : 5;
#pragma unroll
    for (int s = 0; s < LOG; s++) {
        const int c = V >> s, o = 16 >> s;
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < c / 2; j++) {
            const float send = upper ? v[j] : v[j + c / 2];
            const float keep = upper ? v[j + c / 2] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float r = v[0];
#pragma unroll
    for (int o = 16 >> LOG; o >= 1; o >>= 1) r += __shfl_xor_sync(0xffffffffu, r, o);
    return r;
}

// Streaming design.  A CTA owns the contiguous rows [r0, r1) of W, which are
// one contiguous byte range in HBM.  One thread streams that range through a
// ring of NS shared-memory stages with TMA bulk copies (cp.async.bulk), so
// tens of KB per CTA are in flight no matter how many registers the compute
// warps use; the compute threads read their piece of each row from shared
// memory.  Stage c holds rows [r0 + c*SR, r0 + (c+1)*SR) (SR = G*R rows, G
// sub-groups of R rows); the copy starts at the 16-byte boundary at or below
// the stage's first byte, so shared memory keeps each byte's address modulo 16
// and the same aligned loads work on it.  A tail that ends off a 16-byte
// boundary at the very end of the view is copied byte by byte (never past the
// view).  Per-row results go to shared-memory accumulators with atomics, so
// no block barrier sits in the row loop.
constexpr int MMVQ_STAGES = 4;

struct MmvqShape {
    int64_t rows_per_cta;
    int sub_groups;  // G
    int stage_bytes;
};

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(tc::smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(tc::smem_u32(bar))
                 : "memory");
}

template <int WT, int M, int R, int MAXT>
__global__ void __launch_bounds__(MAXT) mmvq_kernel(const uint8_t *__restrict__ w, int64_t n, int64_t k, int64_t rb,
                                                   const uint8_t *__restrict__ xq, int m_act, void *__restrict__ y,
                                                   int yt, int64_t ldy, MmvqShape shp) {
    constexpr int V = R * M;
    constexpr int LOG = V == 1 ? 0 : V == 2 ? 1 : V == 4 ? 2 : V == 8 ? 3 : V == 16 ? 4 : 5;
    static_assert((1 << LOG) == V && V <= 32, "R*M must be a power of two <= 32");
    extern __shared__ __align__(128) uint8_t smem_raw[];
    const int SB = shp.stage_bytes;  // multiple of 16
    uint8_t *stage = smem_raw;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem_raw + MMVQ_STAGES * SB);
    uint64_t *empty = full + MMVQ_STAGES;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + MMVQ_STAGES);
    float *s_acc = reinterpret_cast<float *>(empty + MMVQ_STAGES + 2);  // [rows_per_cta][M]

    const int tid = threadIdx.x, lane = tid & 31, nwarps = blockDim.x >> 5;
    const int64_t P = k / 32;
    const int64_t xrb = P * Q8_1_BYTES;
    const int64_t r0 = (int64_t)blockIdx.x * shp.rows_per_cta;
    const int64_t r1 = r0 + shp.rows_per_cta < n ? r0 + shp.rows_per_cta : n;
    const int64_t SR = (int64_t)shp.sub_groups * R;
    const int nst = (int)((r1 - r0 + SR - 1) / SR);  // stages of this CTA
    const int64_t piece = tid;
    const bool valid = piece < P;
    const uintptr_t wbase = reinterpret_cast<uintptr_t>(w);
    const uintptr_t wend = wbase + (uintptr_t)(n * rb);

    if (tid == 0) {
        for (int s = 0; s < MMVQ_STAGES; s++) {
            tc::mbar_init(&full[s], 1);
            tc::mbar_init(&empty[s], nwarps);
        }
        *abort_flag = 0;
        tc::fence_barrier_init();
    }
    __syncthreads();
    // the next kernel on the stream may launch now; weights never change, so
    // their streaming starts before waiting for the previous kernel
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // stage c: byte range [g0, g1) of the view, copied from a16 = g0 rounded down to 16
    auto issue = [&](int c) {
        const int s = c % MMVQ_STAGES;
        const int64_t ra = r0 + (int64_t)c * SR;
        const int64_t rz = ra + SR < r1 ? ra + SR : r1;
        const uintptr_t g0 = wbase + (uintptr_t)(ra * rb), g1 = wbase + (uintptr_t)(rz * rb);
        const uintptr_t a16 = g0 & ~uintptr_t(15);
        const uintptr_t b16 = (g1 + 15) & ~uintptr_t(15);
        const uintptr_t bulk_end = b16 <= wend ? b16 : (wend & ~uintptr_t(15));
        uint8_t *dst = stage + s * SB;
        const uint32_t bytes = (uint32_t)(bulk_end - a16);
        // the view's last bytes when it does not end on a 16-byte boundary
        // (written before the arrive below publishes the stage)
        for (uintptr_t p = bulk_end; p < g1; p++) dst[p - a16] = *reinterpret_cast<const uint8_t *>(p);
        tc::mbar_arrive_expect_tx(&full[s], bytes);
        if (bytes) bulk_g2s(dst, reinterpret_cast<const void *>(a16), bytes, &full[s]);
    };
    if (tid == 0) {
        for (int c = 0; c < MMVQ_STAGES && c < nst; c++) issue(c);
    }

    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int i = tid; i < shp.rows_per_cta * M; i += blockDim.x) s_acc[i] = 0.0f;
    ActPiece<M> act;
    load_act<WT, M>(act, xq, xrb, m_act, valid ? piece : 0, valid);
    __syncthreads();

    for (int c = 0; c < nst; c++) {
        const int s = c % MMVQ_STAGES;
        const uint32_t ph = (uint32_t)(c / MMVQ_STAGES) & 1u;
        if (*abort_flag) break;
        if (!tc::mbar_wait(&full[s], ph)) { *abort_flag = 1; break; }
        const int64_t ra = r0 + (int64_t)c * SR;
        const uintptr_t a16 = (wbase + (uintptr_t)(ra * rb)) & ~uintptr_t(15);
        // shared-memory address of global byte p is stage + s*SB + (p - a16)
        const uint8_t *srow0 = stage + s * SB + ((wbase + (uintptr_t)(ra * rb)) - a16);
        for (int g = 0; g < shp.sub_groups; g++) {
            const int64_t g0 = ra + (int64_t)g * R;
            if (g0 >= r1) break;
            WPiece<WT> wp[R];
#pragma unroll
            for (int r = 0; r < R; r++) {
                const int64_t rr = g0 + r < r1 ? (int64_t)g * R + r : (r1 - 1 - ra);  // stay inside the stage
                if (valid) load_w<WT>(wp[r], srow0 + rr * rb, piece);
            }
            float part[V];
#pragma unroll
            for (int i = 0; i < V; i++) part[i] = 0.0f;
            if (valid) {
#pragma unroll
                for (int r = 0; r < R; r++) {
                    float acc[M];
#pragma unroll
                    for (int mm = 0; mm < M; mm++) acc[mm] = 0.0f;
                    dot_piece<WT, M>(wp[r], act, piece, acc);
#pragma unroll
                    for (int mm = 0; mm < M; mm++) part[r * M + mm] = acc[mm];
                }
            }
            const float tot = butterfly<V>(part, lane);
            if ((lane & ((32 >> LOG) - 1)) == 0) {
                const int idx = lane >> (5 - LOG);
                const int r = idx / M, mm = idx % M;
                if (g0 + r < r1) atomicAdd(&s_acc[(g0 - r0 + r) * M + mm], tot);
            }
        }
        // this warp is done reading stage s
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(&empty[s]);
        if (tid == 0 && c + MMVQ_STAGES < nst) {
            if (!tc::mbar_wait(&empty[s], ph)) { *abort_flag = 1; }
            else issue(c + MMVQ_STAGES);
        }
    }
    // copies still in flight (only after an abort) land before the CTA exits
    if (tid == 0 && *abort_flag) {
        for (int c = 0; c < nst; c++) tc::mbar_wait(&full[c % MMVQ_STAGES], (uint32_t)(c / MMVQ_STAGES) & 1u);
    }
    __syncthreads();
    const int64_t nr = r1 - r0;
    for (int64_t i = tid; i < nr * M; i += blockDim.x) {
        const int64_t mm = i / nr, r = i - mm * nr;
        if (mm < m_act) store_out(y, yt, mm * ldy + r0 + r, s_acc[r * M + mm]);
    }
}

template <int WT, int M, int R, int MAXT>
inline cudaError_t launch_mmvq_t(const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, void *y,
                                 int yt, int64_t ldy, cudaStream_t s) {
    const int64_t P = k / 32;
    const int nthr = (int)(((P + 31) / 32) * 32);
    const int64_t rb = k / block_elems(WT) * block_bytes(WT);
    auto kern = mmvq_kernel<WT, M, R, MAXT>;
    // stage = G sub-groups of R rows, about 16 KB
    int G = (int)(16384 / (R * rb));
    if (G < 1) G = 1;
    if (G > 8) G = 8;
    const int stage_bytes = (int)(((G * R * rb + 32) + 15) / 16 * 16);
    // one wave of CTAs, each owning a contiguous range of rows
    const int64_t groups = (n + R - 1) / R;
    const int sms = device_info().sm_count;
    const size_t fixed = (size_t)MMVQ_STAGES * stage_bytes + 8 * (2 * MMVQ_STAGES + 2);
    // raise the dynamic shared-memory limit before asking for the occupancy
    // (the query counts a kernel whose request exceeds the limit as unlaunchable)
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(device_info().smem_optin));
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, nthr, fixed + 4096);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)sms * per_sm;
    if (grid > groups) grid = groups;
    const int64_t rows_per_cta = (groups + grid - 1) / grid * R;
    grid = (n + rows_per_cta - 1) / rows_per_cta;
    MmvqShape shp{rows_per_cta, G, stage_bytes};
    const size_t smem = fixed + (size_t)rows_per_cta * M * sizeof(float);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)nthr);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, w, n, k, rb, xq, (int)m, y, yt, ldy, shp);
}

// Threads per CTA = pieces per row (rounded to a warp): K <= 8192 fits in 256
// threads with the full register budget; longer rows use 512-thread CTAs.
// Rows per sub-group R: the default keeps R * M = 16 (8 for m = 1); rows
// longer than 3 KB use R = 1 so that a stage stays within ~20 KB of shared
// memory.  Threads per CTA = pieces per row rounded to a warp: K <= 8192 fits
// 256-thread CTAs with the full register budget, longer rows use 512.
template <int WT, int MAXT>
inline cudaError_t launch_mmvq_mt(const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, void *y,
                                  int yt, int64_t ldy, cudaStream_t s) {
    const int64_t rb = k / block_elems(WT) * block_bytes(WT);
    if (MAXT == 256 && rb <= 3072) {
        if (m <= 1) return launch_mmvq_t<WT, 1, 8, MAXT>(w, n, k, xq, m, y, yt, ldy, s);
        if (m <= 2) return launch_mmvq_t<WT, 2, 8, MAXT>(w, n, k, xq, m, y, yt, ldy, s);
        if (m <= 4) return launch_mmvq_t<WT, 4, 4, MAXT>(w, n, k, xq, m, y, yt, ldy, s);
        return launch_mmvq_t<WT, 8, 2, MAXT>(w, n, k, xq, m, y, yt, ldy, s);
    }
    if (m <= 1) return launch_mmvq_t<WT, 1, 1, MAXT>(w, n, k, xq, m, y, yt, ldy, s);
    if (m <= 2) return launch_mmvq_t<WT, 2, 1, MAXT>(w, n, k, xq, m, y, yt, ldy, s);
    if (m <= 4) return launch_mmvq_t<WT, 4, 1, MAXT>(w, n, k, xq, m, y, yt, ldy, s);
    return launch_mmvq_t<WT, 8, 1, MAXT>(w, n, k, xq, m, y, yt, ldy, s);
}

template <int WT>
inline cudaError_t launch_mmvq_type(const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, void *y,
                                    int yt, int64_t ldy, cudaStream_t s) {
    if (k <= 8192) return launch_mmvq_mt<WT, 256>(w, n, k, xq, m, y, yt, ldy, s);
    return launch_mmvq_mt<WT, 512>(w, n, k, xq, m, y, yt, ldy, s);
}

cudaError_t launch_mmvq_q8_0(const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, void *y, int yt,
                             int64_t ldy, cudaStream_t s);
cudaError_t launch_mmvq_q4_k(const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, void *y, int yt,
                             int64_t ldy, cudaStream_t s);
cudaError_t launch_mmvq_q6_k(const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, void *y, int yt,
                             int64_t ldy, cudaStream_t s);

}  // namespace gg
