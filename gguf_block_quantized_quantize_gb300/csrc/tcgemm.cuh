// Persistent, warp-specialized tcgen05 GEMM shared by the dense MMQ and the
// two MoE mul_mat_id GEMMs:  D[128 weight rows][BN activation rows] += W . X^T
// over K, fp32 accumulators in TMEM.
//
// Operands (all fp16, K-major, 128-byte swizzled rows of 64 values):
//   A = weight rows, unpacked in registers from the packed GGUF blocks
//       (unpack.cuh) by 8 producer warps, each thread half a row per K-step;
//   B = activation rows (the fp16 form d16 * q of q8_1 values), loaded by TMA
//       (dense) or gathered row by row with cp.async (MoE).
// Precision modes:
//   FAST    one fp16 operand per side (packed-half unpack for 16-bit outputs);
//           the product differs from the exact blockwise value by two fp16
//           roundings (about 3e-4 of the row rms);
//   PRECISE hi + lo fp16 operands on both sides (hi = fp16(v), lo = fp16(v - hi))
//           and three MMAs per K step, A_hi B_hi + A_hi B_lo + A_lo B_hi: the
//           result matches the exact blockwise value to about 1e-6.  Used for
//           fp32 outputs and for the MoE intermediate, which is re-quantized.
// Roles (448 threads):
//   warp 0      B producer (TMA: one elected lane; gather: all 32 lanes)
//   warp 1      TMEM allocator + the MMA-issuing thread (two accumulators)
//   warps 2-9   A producers
//   warps 10-13 epilogue (TMEM lane quadrant = warp % 4), overlapping the next
//               tile's mainloop
// Every wait is bounded (1 s); a timeout sets the error word and the CTA exits.
#pragma once

#include <cudaTypedefs.h>

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"
#include "unpack.cuh"

namespace gg {

constexpr int TG_BM = 128;
constexpr int TG_BK = 64;
constexpr int TG_PRODUCERS = 256;
constexpr int TG_THREADS = 64 + TG_PRODUCERS + 128;
constexpr int TG_A_BYTES = TG_BM * TG_BK * 2;  // one fp16 operand tile, 16 KB

enum { TG_DENSE = 0, TG_MOE_GATE_UP = 1, TG_MOE_DOWN = 2 };

struct TgParams {
    // weights
    const uint8_t *w;
    int64_t expert_stride, rb, n, k;
    int64_t kx;  // activation operand row length: k, plus the Q4_K min-term correction columns
    // dense tiles
    int64_t m;
    int tiles_n, tiles_m, tiles_total, ks_per_split;
    void *y;
    int yt;
    int64_t ldy;
    float *yacc;  // split-K partial sums [m][n] (dense) or the MoE output accumulator [T][n] (down)
    // gathered activation rows (MoE)
    const uint16_t *xh, *xl;
    int64_t top_k;
    const int32_t *route_list, *offsets, *counts, *tile_expert, *tile_start, *n_tiles;
    const float *route_w;
    int tiles_x;
    // gate_up outputs (any may be null)
    uint8_t *hq;
    uint16_t *hbf, *h16, *h16lo;
    int64_t hpitch;  // row length of h16 / h16lo: I, plus correction columns when the down weights are Q4_K
};

template <int BN, bool PRECISE>
struct TgShape {
    static constexpr int OPS = PRECISE ? 2 : 1;
    static constexpr int A_STAGE = OPS * TG_A_BYTES;
    static constexpr int B_STAGE = OPS * BN * TG_BK * 2;
    static constexpr int XBUF = 64 * 32 * 4;  // gate_up exchange: 64 rows x 32 columns of fp32
    static constexpr int STAGES_RAW = (200 * 1024 - XBUF) / (A_STAGE + B_STAGE);
    static constexpr int STAGES = STAGES_RAW > 6 ? 6 : STAGES_RAW;
    static constexpr int SMEM = 1024 + STAGES * (A_STAGE + B_STAGE) + XBUF + 512 + BN * 8;
    static constexpr int TMEM_COLS = 2 * BN < 32 ? 32 : 2 * BN;
};

__device__ __forceinline__ void tg_cp_async16(uint32_t dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void tg_cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void tg_cp_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }
__device__ __forceinline__ void tg_named_bar(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Work decomposition of tile t.
struct TgTile {
    int64_t row0;       // first weight row of the 128-row tile (gate_up: first gate row; up rows follow I later)
    int64_t m0;         // dense: first activation row
    int k0, k1;         // K-step range
    int e, route0, n_eff;  // MoE: expert, first route slot in route_list, routes in the tile
};

template <int MODE, int BN>
__device__ __forceinline__ TgTile tg_tile(const TgParams &p, int t, int KS) {
    TgTile d{};
    if (MODE == TG_DENSE) {
        const int nm = p.tiles_n * p.tiles_m;
        d.row0 = (int64_t)(t % p.tiles_n) * TG_BM;
        d.m0 = (int64_t)((t / p.tiles_n) % p.tiles_m) * BN;
        d.k0 = (t / nm) * p.ks_per_split;
        d.k1 = d.k0 + p.ks_per_split < KS ? d.k0 + p.ks_per_split : KS;
        d.n_eff = BN;
    } else {
        const int tx = t % p.tiles_x, tl = t / p.tiles_x;
        d.e = p.tile_expert[tl];
        const int s0 = p.tile_start[tl];
        const int cnt = p.counts[d.e];
        d.n_eff = cnt - s0 < BN ? cnt - s0 : BN;
        d.route0 = p.offsets[d.e] + s0;
        d.row0 = MODE == TG_MOE_GATE_UP ? (int64_t)tx * 64 : (int64_t)tx * TG_BM;
        d.k0 = 0;
        d.k1 = KS;
    }
    return d;
}

template <int WT, int BN, bool PRECISE, int MODE, int OT>
__global__ void __launch_bounds__(TG_THREADS, 1)
    tg_kernel(const __grid_constant__ CUtensorMap map_hi, const __grid_constant__ CUtensorMap map_lo, const TgParams p,
              int *err) {
    using S = TgShape<BN, PRECISE>;
    constexpr int ST = S::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sA = smem;                             // [ST][OPS][16 KB]
    uint8_t *sB = smem + ST * S::A_STAGE;           // [ST][OPS][BN * 128]
    float *xbuf = reinterpret_cast<float *>(sB + ST * S::B_STAGE);
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(xbuf) + S::XBUF);
    uint64_t *full_a = bars, *full_b = bars + ST, *empty = bars + 2 * ST;
    uint64_t *tfull = bars + 3 * ST, *tempty = bars + 3 * ST + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(bars + 3 * ST + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int KS = (int)((p.kx + TG_BK - 1) / TG_BK);      // K steps of the product
    const int KS_W = (int)((p.k + TG_BK - 1) / TG_BK);     // K steps that hold weight values
    const int tiles_total = MODE == TG_DENSE ? p.tiles_total : *p.n_tiles * p.tiles_x;
    constexpr bool H2 = !PRECISE && OT != GGUF_F32 && MODE == TG_DENSE;

    if (tid == 0) {
        for (int s = 0; s < ST; s++) {
            tc::mbar_init(&full_a[s], TG_PRODUCERS);
            tc::mbar_init(&full_b[s], MODE == TG_DENSE ? 1 : 32);
            tc::mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], 128);
        }
        *abort_flag = 0;
        tc::fence_barrier_init();
        if (MODE == TG_DENSE) {
            tc::prefetch_tmap(&map_hi);
            if (PRECISE) tc::prefetch_tmap(&map_lo);
        }
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, S::TMEM_COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto fail = [&](int code) {
        *abort_flag = 1;
        atomicOr(err, code);
    };

    if (warp == 0) {
        // ================= B producer
        if (MODE == TG_DENSE) {
            if (lane == 0) {
                int it = 0, last = 0;
                for (int t = blockIdx.x; t < tiles_total && !*abort_flag; t += gridDim.x) {
                    const TgTile d = tg_tile<MODE, BN>(p, t, KS);
                    for (int ks = d.k0; ks < d.k1; ks++, it++) {
                        const int s = it % ST;
                        const uint32_t ph = (uint32_t)(it / ST) & 1u;
                        if (*abort_flag) break;
                        if (!tc::mbar_wait(&empty[s], ph ^ 1u)) { fail(1); break; }
                        tc::mbar_arrive_expect_tx(&full_b[s], (uint32_t)S::B_STAGE);
                        uint8_t *dst = sB + s * S::B_STAGE;
                        tc::tma_load_2d(dst, &map_hi, &full_b[s], ks * TG_BK, (int32_t)d.m0);
                        if (PRECISE) tc::tma_load_2d(dst + BN * TG_BK * 2, &map_lo, &full_b[s], ks * TG_BK, (int32_t)d.m0);
                        last = it + 1;
                    }
                }
                if (*abort_flag)  // copies already issued land before the CTA exits
                    for (int i = last - ST < 0 ? 0 : last - ST; i < last; i++)
                        tc::mbar_wait(&full_b[i % ST], (uint32_t)(i / ST) & 1u);
            }
        } else {
            // gather: lane handles rows lane, lane + 32, ... of the tile
            constexpr int RPL = (BN + 31) / 32;
            constexpr int LAG = 2;  // cp.async groups in flight per lane
            int it = 0;
            for (int t = blockIdx.x; t < tiles_total && !*abort_flag; t += gridDim.x) {
                const TgTile d = tg_tile<MODE, BN>(p, t, KS);
                int64_t srow[RPL];
#pragma unroll
                for (int i = 0; i < RPL; i++) {
                    const int j = lane + 32 * i;
                    const int r = (j < BN && j < d.n_eff) ? p.route_list[d.route0 + j] : -1;
                    srow[i] = r < 0 ? -1 : (MODE == TG_MOE_GATE_UP ? r / p.top_k : r);
                }
                const int it0 = it;
                for (int ks = 0; ks < KS; ks++, it++) {
                    const int s = it % ST;
                    const uint32_t ph = (uint32_t)(it / ST) & 1u;
                    if (*abort_flag) break;
                    if (!tc::mbar_wait(&empty[s], ph ^ 1u)) { fail(1); break; }
                    const uint32_t bbase = tc::smem_u32(sB + s * S::B_STAGE);
#pragma unroll
                    for (int i = 0; i < RPL; i++) {
                        const int j = lane + 32 * i;
                        if (j >= BN) continue;
#pragma unroll
                        for (int c = 0; c < 8; c++) {
                            const int64_t kk = (int64_t)ks * TG_BK + 8 * c;
                            const bool v = srow[i] >= 0 && kk < p.kx;
                            const uint32_t off = (uint32_t)(j * 128 + ((c ^ (j & 7)) * 16));
                            tg_cp_async16(bbase + off, v ? (const void *)(p.xh + srow[i] * p.kx + kk) : (const void *)p.xh,
                                          v ? 16u : 0u);
                            if (PRECISE)
                                tg_cp_async16(bbase + BN * TG_BK * 2 + off,
                                              v ? (const void *)(p.xl + srow[i] * p.kx + kk) : (const void *)p.xl,
                                              v ? 16u : 0u);
                        }
                    }
                    tg_cp_commit();
                    if (it - it0 >= LAG) {
                        tg_cp_wait<LAG>();
                        tc::fence_proxy_async_smem();
                        tc::mbar_arrive(&full_b[(it - LAG) % ST]);
                    }
                }
                tg_cp_wait<0>();
                tc::fence_proxy_async_smem();
                for (int i = (it - LAG > it0 ? it - LAG : it0); i < it; i++) tc::mbar_arrive(&full_b[i % ST]);
            }
        }
    } else if (warp == 1) {
        // ================= MMA issuer
        if (lane == 0) {
            int it = 0, i = 0;
            for (int t = blockIdx.x; t < tiles_total; t += gridDim.x, i++) {
                const TgTile d = tg_tile<MODE, BN>(p, t, KS);
                const int b = i & 1;
                if (*abort_flag) break;
                if (!tc::mbar_wait(&tempty[b], ((uint32_t)(i >> 1) & 1u) ^ 1u)) { fail(16); break; }
                tc::tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * BN);
                const int n_mma = MODE == TG_DENSE ? BN : ((d.n_eff + 15) / 16) * 16;
                const uint32_t idesc = tc::idesc_f16_f32(TG_BM, n_mma);
                for (int ks = d.k0; ks < d.k1; ks++, it++) {
                    const int s = it % ST;
                    const uint32_t ph = (uint32_t)(it / ST) & 1u;
                    if (*abort_flag) break;
                    if (!tc::mbar_wait(&full_a[s], ph) || !tc::mbar_wait(&full_b[s], ph)) { fail(2); break; }
                    tc::tc_fence_after();
                    const uint32_t a0 = tc::smem_u32(sA + s * S::A_STAGE);
                    const uint32_t b0 = tc::smem_u32(sB + s * S::B_STAGE);
#pragma unroll
                    for (int kk = 0; kk < TG_BK / 16; kk++) {
                        const uint32_t acc_in = (ks != d.k0 || kk != 0) ? 1u : 0u;
                        tc::mma_f16(acc, tc::sw128_desc(a0 + 32 * kk), tc::sw128_desc(b0 + 32 * kk), idesc, acc_in);
                        if (PRECISE) {
                            tc::mma_f16(acc, tc::sw128_desc(a0 + 32 * kk),
                                        tc::sw128_desc(b0 + BN * TG_BK * 2 + 32 * kk), idesc, 1u);
                            tc::mma_f16(acc, tc::sw128_desc(a0 + TG_A_BYTES + 32 * kk), tc::sw128_desc(b0 + 32 * kk),
                                        idesc, 1u);
                        }
                    }
                    tc::mma_commit(&empty[s]);
                }
                tc::mma_commit(&tfull[b]);
            }
        }
    } else if (warp < 2 + TG_PRODUCERS / 32) {
        // ================= A producers: thread p -> row p % 128, half p / 128
        const int pidx = tid - 64;
        const int r = pidx & (TG_BM - 1), half = pidx >> 7;
        int it = 0;
        for (int t = blockIdx.x; t < tiles_total && !*abort_flag; t += gridDim.x) {
            const TgTile d = tg_tile<MODE, BN>(p, t, KS);
            int64_t row;
            if (MODE == TG_MOE_GATE_UP) row = r < 64 ? d.row0 + r : p.n / 2 + d.row0 + (r - 64);
            else row = d.row0 + r;
            const bool live = row < p.n;
            const uint8_t *wrow = p.w + (MODE == TG_DENSE ? 0 : (int64_t)d.e * p.expert_stride) + (live ? row : 0) * p.rb;
            KHalf<WT> u0, u1;
            if constexpr (WT == GGUF_Q8_0) { u0.kblocks = p.k / 32; u1.kblocks = p.k / 32; }
            const int kw1 = d.k1 < KS_W ? d.k1 : KS_W;  // weight K steps of this tile
            if (live) {
                if (d.k0 < kw1) u0.load(wrow, d.k0, half);
                if (d.k0 + 1 < kw1) u1.load(wrow, d.k0 + 1, half);
            }
            // one K step: unpack (weight steps) or the min-term correction values
            // dmin * m_j of 32 sub-blocks (Q4_K steps past the weights), then store
            auto produce = [&](const KHalf<WT> &u, int ks) -> bool {
                const int s = it % ST;
                const uint32_t ph = (uint32_t)(it / ST) & 1u;
                it++;
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int i = 0; i < 16; i++) { hi[i] = 0u; lo[i] = 0u; }
                if (live && ks < KS_W) {
                    if (H2) u.unpack_h2(ks, half, hi);
                    else {
                        float v[32];
                        u.unpack_f32(ks, half, v);
                        if (PRECISE) pack_split(v, hi, lo);
                        else pack_single(v, hi);
                    }
                } else if (live && WT == GGUF_Q4_K) {
                    const int64_t j0 = (int64_t)ks * TG_BK - p.k + 32 * half;  // first sub-block of this half
                    const int64_t nsub = p.k / 32;
                    float v[32];
#pragma unroll
                    for (int g4 = 0; g4 < 4; g4++) {  // 8 sub-blocks per super-block header
                        const int64_t sb = j0 / 8 + g4;
                        uint4 hdr = make_uint4(0, 0, 0, 0);
                        if (sb * 8 < nsub) hdr = *reinterpret_cast<const uint4 *>(wrow + sb * Q4_K_BYTES);
                        const uint32_t sc[3] = {hdr.y, hdr.z, hdr.w};
                        const float dmin = h2f(hdr.x >> 16);
#pragma unroll
                        for (int jj = 0; jj < 8; jj++) {
                            int sv, mv;
                            q4k_scale_min(sc, jj, sv, mv);
                            v[8 * g4 + jj] = (sb * 8 + jj < nsub) ? __fmul_rn(dmin, (float)mv) : 0.0f;
                        }
                    }
                    pack_single(v, hi);
                }
                if (*abort_flag) return false;
                if (!tc::mbar_wait(&empty[s], ph ^ 1u)) { fail(4); return false; }
                store_sw128_half(sA + s * S::A_STAGE, r, half, hi);
                if (PRECISE) store_sw128_half(sA + s * S::A_STAGE + TG_A_BYTES, r, half, lo);
                tc::fence_proxy_async_smem();
                tc::mbar_arrive(&full_a[s]);
                return true;
            };
            bool ok = true;
            for (int ks = d.k0; ks < d.k1 && ok; ks += 2) {
                ok = produce(u0, ks);
                if (live && ks + 2 < kw1) u0.load(wrow, ks + 2, half);  // two K-steps ahead
                if (ok && ks + 1 < d.k1) {
                    ok = produce(u1, ks + 1);
                    if (live && ks + 3 < kw1) u1.load(wrow, ks + 3, half);
                }
            }
            if (!ok) break;
        }
    } else {
        // ================= epilogue
        const int q = warp & 3;
        int i = 0;
        for (int t = blockIdx.x; t < tiles_total; t += gridDim.x, i++) {
            const TgTile d = tg_tile<MODE, BN>(p, t, KS);
            const int b = i & 1;
            const bool ok = tc::mbar_wait(&tfull[b], (uint32_t)(i >> 1) & 1u);
            if (!ok) fail(8);
            tc::tc_fence_after();
            const bool go = ok && !*abort_flag;
            if (MODE == TG_DENSE) {
                const int64_t orow = d.row0 + 32 * q + lane;
#pragma unroll 1
                for (int c = 0; c * 32 < BN && go; c++) {
                    uint32_t rr[32];
                    tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * BN + 32 * c), rr);
                    tc::tmem_ld_wait();
                    if (orow < p.n) {
#pragma unroll
                        for (int jj = 0; jj < 32; jj++) {
                            const int64_t mm = d.m0 + 32 * c + jj;
                            if (32 * c + jj < BN && mm < p.m) {
                                if (p.yacc) atomicAdd(&p.yacc[mm * p.n + orow], __uint_as_float(rr[jj]));
                                else store_out(p.y, OT, mm * p.ldy + orow, __uint_as_float(rr[jj]));
                            }
                        }
                    }
                }
            } else if (MODE == TG_MOE_DOWN) {
                const int64_t orow = d.row0 + 32 * q + lane;
#pragma unroll 1
                for (int c = 0; c * 32 < d.n_eff && go; c++) {
                    uint32_t rr[32];
                    tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * BN + 32 * c), rr);
                    tc::tmem_ld_wait();
                    if (orow < p.n) {
#pragma unroll 4
                        for (int jj = 0; jj < 32; jj++) {
                            const int j = 32 * c + jj;
                            if (j < d.n_eff) {
                                const int rt = p.route_list[d.route0 + j];
                                const float wgt = p.route_w ? p.route_w[rt] : 1.0f;
                                atomicAdd(&p.yacc[(int64_t)(rt / p.top_k) * p.n + orow], wgt * __uint_as_float(rr[jj]));
                            }
                        }
                    }
                }
            } else {
                // gate rows in TMEM lanes 0..63 (q = 0, 1), up rows in 64..127 (q = 2, 3)
                const int64_t idim = p.n / 2;
                const int64_t hrb = idim / 32 * Q8_1_BYTES;
                const int il = 32 * (q & 1) + lane;          // i within the 64-row slice
                const int64_t icol = d.row0 + il;             // column of h
#pragma unroll 1
                for (int c = 0; c * 32 < BN; c++) {
                    const bool any = go && 32 * c < d.n_eff;  // uniform across the 4 warps
                    uint32_t rr[32];
                    if (any) {
                        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * BN + 32 * c), rr);
                        tc::tmem_ld_wait();
                        if (q >= 2) {
#pragma unroll
                            for (int jj = 0; jj < 32; jj++) xbuf[jj * 64 + il] = __uint_as_float(rr[jj]);
                        }
                    }
                    tg_named_bar(1, 128);
                    if (any && q < 2) {
#pragma unroll 1
                        for (int jj = 0; jj < 32; jj++) {
                            const int j = 32 * c + jj;
                            if (j >= d.n_eff) break;
                            const int64_t rt = p.route_list[d.route0 + j];
                            const float gv = __uint_as_float(rr[jj]);
                            const float uv = xbuf[jj * 64 + il];
                            const float hf = gv / (1.0f + expf(-gv)) * uv;
                            const uint16_t hb = f2bf_rn(hf);
                            const float hx = bf2f(hb);  // the intermediate in the activation dtype
                            if (p.hbf) p.hbf[rt * idim + icol] = hb;
                            float amax = fabsf(hx);
#pragma unroll
                            for (int o = 16; o >= 1; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
                            const float dq = __fdiv_rn(amax, 127.0f);
                            const int qv = dq != 0.0f ? (int)roundf(__fdiv_rn(hx, dq)) : 0;
                            int sum = qv;
#pragma unroll
                            for (int o = 16; o >= 1; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
                            const uint16_t dh = f2h_rn(dq);
                            if (p.hq) {
                                uint8_t *blk = p.hq + rt * hrb + (icol / 32) * Q8_1_BYTES;
                                blk[4 + lane] = (uint8_t)(int8_t)qv;
                                if (lane == 0) {
                                    const uint16_t sh = f2h_rn(__fmul_rn(dq, (float)sum));
                                    *reinterpret_cast<uint32_t *>(blk) = (uint32_t)dh | ((uint32_t)sh << 16);
                                }
                            }
                            if (p.h16) {
                                const float v = h2f(dh) * (float)qv;
                                const uint16_t vh = f2h_rn(v);
                                p.h16[rt * p.hpitch + icol] = vh;
                                if (p.h16lo) p.h16lo[rt * p.hpitch + icol] = f2h_rn(v - h2f(vh));
                                if (p.hpitch > idim) {
                                    // min-term correction column of this q8_1 block (Q4_K down weights),
                                    // and the zero padding of the row (written once, by the first column tile)
                                    if (lane == 0) {
                                        const uint16_t sh = f2h_rn(__fmul_rn(dq, (float)sum));
                                        p.h16[rt * p.hpitch + idim + icol / 32] = f2h_rn(h2f(dh) * (float)sum - h2f(sh));
                                        if (p.h16lo) p.h16lo[rt * p.hpitch + idim + icol / 32] = 0;
                                    }
                                    if (d.row0 == 0 && q == 0)
                                        for (int64_t c2 = idim + idim / 32 + lane; c2 < p.hpitch; c2 += 32) {
                                            p.h16[rt * p.hpitch + c2] = 0;
                                            if (p.h16lo) p.h16lo[rt * p.hpitch + c2] = 0;
                                        }
                                }
                            }
                        }
                    }
                    tg_named_bar(1, 128);
                }
            }
            tc::tc_fence_before();
            tc::mbar_arrive(&tempty[b]);
            if (!ok) break;
        }
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 1) tc::tmem_dealloc(tmem, S::TMEM_COLS);
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// fp16 rows [rows][k] as a TMA tensor map with a 64 x bn box (128-byte swizzle)
inline cudaError_t tg_make_map(CUtensorMap *map, const uint16_t *base, int64_t rows, int64_t k, int bn) {
    auto enc = tensor_map_encoder();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t gdim[2] = {(cuuint64_t)k, (cuuint64_t)rows};
    cuuint64_t gstride[1] = {(cuuint64_t)k * 2};
    cuuint32_t box[2] = {(cuuint32_t)TG_BK, (cuuint32_t)bn};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<uint16_t *>(base), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

int *tg_error_word();

template <int WT, int BN, bool PRECISE, int MODE, int OT>
inline cudaError_t tg_launch(const CUtensorMap &mh, const CUtensorMap &ml, const TgParams &p, int grid,
                             cudaStream_t s) {
    using S = TgShape<BN, PRECISE>;
    auto kern = tg_kernel<WT, BN, PRECISE, MODE, OT>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, S::SMEM);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    kern<<<grid, TG_THREADS, S::SMEM, s>>>(mh, ml, p, tg_error_word());
    return cudaGetLastError();
}

}  // namespace gg
