// Persistent, warp-specialized tcgen05 GEMM shared by the dense MMQ and the
// two MoE mul_mat_id GEMMs:  D[128 weight rows][BN activation rows] += W . X^T
// over K, fp32 accumulators in TMEM.
//
// Operands (all fp16, K-major, 128-byte swizzled rows of 64 values):
//   A = weight rows, unpacked in registers from the packed GGUF blocks
//       (unpack.cuh) by 8 producer warps; per K-step a thread takes one part
//       (half or quarter) of one or two rows.  Where the weight rows can be
//       described to TMA (row bytes a multiple of 16, or a few rows together),
//       the packed bytes of 128 rows x one 256-value chunk (or whole short
//       rows) are staged in a ring of shared-memory buffers by bulk tensor
//       copies and the producers unpack from there; otherwise they load the
//       packed bytes from global memory themselves, consecutive lanes sharing
//       a row so that each warp-wide load reads 16 (8) rows of contiguous bytes;
//   B = activation rows (the fp16 form d16 * q of q8_1 values), loaded by TMA:
//       tiles (dense) or tile::gather4 of the routed rows (MoE; 4 rows per copy).
// Precision modes:
//   FAST    one fp16 operand per side (packed-half unpack for 16-bit outputs);
//           the product differs from the exact blockwise value by two fp16
//           roundings (about 3e-4 of the row rms);
//   PRECISE hi + lo fp16 operands on both sides (hi = fp16(v), lo = fp16(v - hi))
//           and three MMAs per K step, A_hi B_hi + A_hi B_lo + A_lo B_hi: the
//           result matches the exact blockwise value to about 1e-6.  Used for
//           fp32 outputs and for the MoE intermediate, which is re-quantized.
// Roles (480 threads):
//   warp 0      B producer (dense: one elected lane; MoE: lane i gathers rows 4i .. 4i+3)
//   warp 1      TMEM allocator + the MMA-issuing thread (two accumulators)
//   warps 2-9   A producers
//   warps 10-13 epilogue (TMEM lane quadrant = warp % 4), overlapping the next
//               tile's mainloop
//   warp 14     packed-weight loader (one elected lane issues the bulk copies)
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
constexpr int TG_GROUPS = 2;   // producer groups, each building every TG_GROUPS-th K-step
constexpr int TG_THREADS = 64 + TG_PRODUCERS + 128 + 32;
constexpr int TG_LOADER_WARP = 14;
constexpr int TG_MAX_PSTAGES = 8;
constexpr int TG_SMEM_MAX = 232448;   // dynamic shared memory a CTA may opt in to

// Packed bytes of one 256-value chunk of a weight row, and the width of the
// 16-byte-aligned window that always covers one (a chunk that starts inside a
// 16-byte word needs up to 16 - gcd(bytes, 16) more).
__host__ __device__ constexpr int tg_chunk_bytes(int wt) {
    return wt == GGUF_Q4_K ? 144 : wt == GGUF_Q5_K ? 176 : wt == GGUF_Q6_K ? 210 : wt == GGUF_Q8_0 ? 272
         : wt == GGUF_Q4_0 ? 144 : wt == GGUF_MXFP4 ? 136 : 0;
}
__host__ __device__ constexpr int tg_chunk_pitch(int wt) {
    return wt == GGUF_Q6_K ? 224 : wt == GGUF_MXFP4 ? 144 : tg_chunk_bytes(wt);
}
constexpr int TG_A_BYTES = TG_BM * TG_BK * 2;  // one fp16 operand tile, 16 KB

enum { TG_DENSE = 0, TG_MOE_GATE_UP = 1, TG_MOE_DOWN = 2 };

struct TgParams {
    // weights
    const uint8_t *w;
    int64_t expert_stride, rb, n, k;
    int64_t kx;  // activation operand row length: k, plus the Q4_K / Q5_K min-term correction columns
    // dense tiles
    int64_t m;
    int tiles_n, tiles_m, tiles_total, ks_per_split;
    int m_fast;   // dense tile order: the activation tile index varies fastest (weights larger than L2)
    void *y;
    int yt;
    int64_t ldy;
    float *yacc;  // split-K partial sums [m][n] (dense), or the MoE down per-route outputs in grouped
                  // order, as ceil(n / 128) blocks [zrows][128]
    float *ysum;  // MoE down with the fused weighted sum: fp32 token rows [T][n], zeroed before the call
    int ysum_bulk;  // 1: the weighted rows are added by bulk reduce-adds (n % 4 == 0, ysum 16-byte aligned);
                    // 0: by scalar fp32 atomics
    int64_t zrows;  // MoE down: rows (routes) of one 128-column block of yacc
    int ystore;     // dense: the output is written by bulk tensor stores through map_y
    // gathered activation rows (MoE)
    const uint16_t *xh, *xl;
    int64_t top_k;
    const int32_t *route_list, *offsets, *counts, *tile_expert, *tile_start, *n_tiles;
    const float *route_w;
    int tiles_x;
    // gate_up outputs (any may be null)
    uint8_t *hq;
    uint16_t *hbf, *h16, *h16lo;
    int64_t hpitch;  // row length of h16 / h16lo: I, plus correction columns when the down weights are Q4_K / Q5_K
    int h16_grouped;  // h16 / h16lo rows in grouped route order (the fused down GEMM's operand); 0: route order
    // staged packed weights (pstages == 0: the producers load from global memory)
    int pstages;         // buffers in the ring
    int pkc;             // K-steps per staged chunk (4: one 256-value chunk; or every weight K-step of a row)
    int pchunked;        // 1: chunks of 256 values in an aligned window; 0: whole rows
    int pgroup;          // rows per line of the tensor map (whole rows whose byte length is not a multiple of 16)
    int64_t ppitch;      // bytes between rows in a buffer
    int64_t pstage_bytes;
    int64_t pb256;       // packed bytes per 256 values
};

template <int WT, int BN, bool PRECISE, int MODE>
struct TgShape {
    static constexpr int OPS = PRECISE ? 2 : 1;
    // tiles of at most 128 activation rows keep the unpacked weight operand in
    // tensor memory (beside the two accumulators); wider tiles in shared memory
    static constexpr bool ATM = BN <= 128;
    static constexpr int A_COL0 = 2 * BN;   // first TMEM column of the A stages
    static constexpr int A_STAGE = ATM ? 0 : OPS * TG_A_BYTES;
    static constexpr int B_STAGE = OPS * BN * TG_BK * 2;
    // gate_up exchange: gate and up values of 64 rows x 32 routes, fp32;
    // down: two 32-route x 128-column fp32 buffers of the bulk output stores;
    // dense: two 32 x 32 output boxes per epilogue warp (fp32 outputs are the
    // precise mode, 16-bit outputs the fast one)
    static constexpr int XBUF = MODE == TG_MOE_GATE_UP ? 2 * 64 * 32 * 4
                              : MODE == TG_MOE_DOWN    ? 2 * 32 * 128 * 4
                                                       : 4 * 2 * 32 * 32 * (PRECISE ? 4 : 2);
    static constexpr int BAR_BYTES = 1024;
    static constexpr int FIXED = 1024 + XBUF + BAR_BYTES + BN * 8;
    // room kept for two buffers of staged packed weights: 128 rows x one chunk
    // window, or (MoE down, fast mode) whole rows of up to 432 bytes
    static constexpr int PCHUNK = (TG_BM * tg_chunk_pitch(WT) + 1023) / 1024 * 1024;
    static constexpr int PRES = (MODE == TG_MOE_DOWN && 2 * PCHUNK < 110592) ? 110592 : 2 * PCHUNK;
    static constexpr int STAGES_RAW = (TG_SMEM_MAX - FIXED - PRES) / (A_STAGE + B_STAGE);
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;   // B stages (and A stages in shared memory)
    static_assert(STAGES >= 2, "at least two operand stages");
    static constexpr int BASE = FIXED + STAGES * (A_STAGE + B_STAGE);   // bytes before the packed ring
    // A stages: in TMEM, OPS x 32 columns each (64 fp16 of K per row)
    static constexpr int STA_RAW = ATM ? (512 - A_COL0) / (32 * OPS) : STAGES;
    static constexpr int STA = STA_RAW > 8 ? 8 : STA_RAW;
    static_assert(STA >= 2, "at least two A stages");
    static constexpr int TMEM_COLS = ATM ? 512 : (2 * BN < 32 ? 32 : 2 * BN);
};

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
        // m_fast: the CTAs of one wave share few weight tiles, each read from DRAM
        // once and from L2 by the CTAs of its other activation tiles
        const int tn = p.m_fast ? (t / p.tiles_m) % p.tiles_n : t % p.tiles_n;
        const int tm = p.m_fast ? t % p.tiles_m : (t / p.tiles_n) % p.tiles_m;
        d.row0 = (int64_t)tn * TG_BM;
        d.m0 = (int64_t)tm * BN;
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
    tg_kernel(const __grid_constant__ CUtensorMap map_hi, const __grid_constant__ CUtensorMap map_lo,
              const __grid_constant__ CUtensorMap map_w, const __grid_constant__ CUtensorMap map_y, const TgParams p,
              int *err) {
    using S = TgShape<WT, BN, PRECISE, MODE>;
    constexpr int ST = S::STAGES, STA = S::STA;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned base, derived from smem_raw by pointer arithmetic so
    // that loads through it compile to shared-memory loads
    uint8_t *smem = smem_raw + ((1024u - (tc::smem_u32(smem_raw) & 1023u)) & 1023u);
    uint8_t *sA = smem;                             // [ST][OPS][16 KB]
    uint8_t *sB = smem + ST * S::A_STAGE;           // [ST][OPS][BN * 128]
    uint8_t *sP = sB + ST * S::B_STAGE;             // [pstages][pstage_bytes] packed weights
    float *xbuf = reinterpret_cast<float *>(sP + (int64_t)p.pstages * p.pstage_bytes);
    uint64_t *bars = reinterpret_cast<uint64_t *>(reinterpret_cast<uint8_t *>(xbuf) + S::XBUF);
    uint64_t *full_a = bars, *empty_a = bars + STA;            // A stages (TMEM or shared memory)
    uint64_t *full_b = bars + 2 * STA, *empty_b = full_b + ST;  // B stages
    uint64_t *tfull = empty_b + ST, *tempty = tfull + 2;
    uint64_t *drain = tfull + 4;  // completion of every MMA this CTA issued
    uint64_t *pfull = drain + 1, *pempty = pfull + TG_MAX_PSTAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(pempty + TG_MAX_PSTAGES);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int KS = (int)((p.kx + TG_BK - 1) / TG_BK);      // K steps of the product
    const int KS_W = (int)((p.k + TG_BK - 1) / TG_BK);     // K steps that hold weight values
    const int tiles_total = MODE == TG_DENSE ? p.tiles_total : *p.n_tiles * p.tiles_x;
    constexpr bool H2 = !PRECISE && OT != GGUF_F32 && MODE == TG_DENSE;

    if (tid == 0) {
        for (int s = 0; s < STA; s++) {
            tc::mbar_init(&full_a[s], TG_PRODUCERS / TG_GROUPS);
            tc::mbar_init(&empty_a[s], 1);
        }
        for (int s = 0; s < ST; s++) {
            tc::mbar_init(&full_b[s], 1);
            tc::mbar_init(&empty_b[s], 1);
        }
        for (int b = 0; b < 2; b++) {
            tc::mbar_init(&tfull[b], 1);
            tc::mbar_init(&tempty[b], 128);
        }
        tc::mbar_init(drain, 1);
        for (int s = 0; s < p.pstages; s++) {
            tc::mbar_init(&pfull[s], 1);
            tc::mbar_init(&pempty[s], TG_PRODUCERS / 32);
        }
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::prefetch_tmap(&map_hi);
        if (PRECISE) tc::prefetch_tmap(&map_lo);
        if (p.pstages > 0) tc::prefetch_tmap(&map_w);
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
        if constexpr (MODE == TG_DENSE) {
            if (lane == 0) {
                int it = 0, last = 0;
                for (int t = blockIdx.x; t < tiles_total && !*abort_flag; t += gridDim.x) {
                    const TgTile d = tg_tile<MODE, BN>(p, t, KS);
                    for (int ks = d.k0; ks < d.k1; ks++, it++) {
                        const int s = it % ST;
                        const uint32_t ph = (uint32_t)(it / ST) & 1u;
                        if (*abort_flag) break;
                        if (!tc::mbar_wait(&empty_b[s], ph ^ 1u)) { fail(1); break; }
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
            // MoE: the operand rows are in grouped (expert-sorted) route order, so
            // a tile's routes are consecutive rows from route0; rows past the
            // expert's routes belong to the next expert and only fill MMA columns
            // the epilogue ignores (rows past the operand read as zeros)
            if (lane == 0) {
                int it = 0, last = 0;
                for (int t = blockIdx.x; t < tiles_total && !*abort_flag; t += gridDim.x) {
                    const TgTile d = tg_tile<MODE, BN>(p, t, KS);
                    for (int ks = 0; ks < KS; ks++, it++) {
                        const int s = it % ST;
                        const uint32_t ph = (uint32_t)(it / ST) & 1u;
                        if (*abort_flag) break;
                        if (!tc::mbar_wait(&empty_b[s], ph ^ 1u)) { fail(1); break; }
                        tc::mbar_arrive_expect_tx(&full_b[s], (uint32_t)S::B_STAGE);
                        uint8_t *dst = sB + s * S::B_STAGE;
                        tc::tma_load_2d(dst, &map_hi, &full_b[s], ks * TG_BK, d.route0);
                        if (PRECISE) tc::tma_load_2d(dst + BN * TG_BK * 2, &map_lo, &full_b[s], ks * TG_BK, d.route0);
                        last = it + 1;
                    }
                }
                if (*abort_flag)  // copies already issued land before the CTA exits
                    for (int i = last - ST < 0 ? 0 : last - ST; i < last; i++)
                        tc::mbar_wait(&full_b[i % ST], (uint32_t)(i / ST) & 1u);
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
                    const int s = it % ST, sa = it % STA;
                    const uint32_t ph = (uint32_t)(it / ST) & 1u, pha = (uint32_t)(it / STA) & 1u;
                    if (*abort_flag) break;
                    if (!tc::mbar_wait(&full_a[sa], pha) || !tc::mbar_wait(&full_b[s], ph)) { fail(2); break; }
                    tc::tc_fence_after();
                    const uint32_t b0 = tc::smem_u32(sB + s * S::B_STAGE);
                    if constexpr (S::ATM) {
                        // A hi (and lo) in TMEM columns of stage sa; 8 columns per K = 16
                        const uint32_t a0 = tmem + (uint32_t)(S::A_COL0 + sa * 32 * S::OPS);
#pragma unroll
                        for (int kk = 0; kk < TG_BK / 16; kk++) {
                            const uint32_t acc_in = (ks != d.k0 || kk != 0) ? 1u : 0u;
                            tc::mma_f16_ts(acc, a0 + 8 * kk, tc::sw128_desc(b0 + 32 * kk), idesc, acc_in);
                            if (PRECISE) {
                                tc::mma_f16_ts(acc, a0 + 8 * kk, tc::sw128_desc(b0 + BN * TG_BK * 2 + 32 * kk), idesc, 1u);
                                tc::mma_f16_ts(acc, a0 + 32 + 8 * kk, tc::sw128_desc(b0 + 32 * kk), idesc, 1u);
                            }
                        }
                    } else {
                        const uint32_t a0 = tc::smem_u32(sA + sa * S::A_STAGE);
#pragma unroll
                        for (int kk = 0; kk < TG_BK / 16; kk++) {
                            const uint32_t acc_in = (ks != d.k0 || kk != 0) ? 1u : 0u;
                            tc::mma_f16(acc, tc::sw128_desc(a0 + 32 * kk), tc::sw128_desc(b0 + 32 * kk), idesc, acc_in);
                            if (PRECISE) {
                                tc::mma_f16(acc, tc::sw128_desc(a0 + 32 * kk),
                                            tc::sw128_desc(b0 + BN * TG_BK * 2 + 32 * kk), idesc, 1u);
                                tc::mma_f16(acc, tc::sw128_desc(a0 + TG_A_BYTES + 32 * kk),
                                            tc::sw128_desc(b0 + 32 * kk), idesc, 1u);
                            }
                        }
                    }
                    tc::mma_commit(&empty_a[sa]);
                    tc::mma_commit(&empty_b[s]);
                }
                tc::mma_commit(&tfull[b]);
            }
            // every MMA issued so far has finished before TMEM is released (after
            // an abort the epilogue no longer waits for them)
            tc::mma_commit(drain);
            if (!tc::mbar_wait(drain, 0)) fail(2);
        }
    } else if (warp < 2 + TG_PRODUCERS / 32) {
      if constexpr (S::ATM) {
        // ================= A producers, operand in TMEM.  Warp w writes the
        // TMEM lane quadrant w % 4: a thread owns tile row 32 * (w % 4) + lane
        // and writes all 64 values of its row per K-step; the 4 warps of group
        // (w - 2) / 4 take the K-steps whose running index is the group
        // modulo TG_GROUPS.
        using U = KQ<WT>;
        constexpr int PARTS = U::PARTS, VW = 8 * U::CHUNKS;
        const int grp = (warp - 2) >> 2;
        const int r = 32 * (warp & 3) + lane;
        const uint32_t tlane = (uint32_t)(32 * (warp & 3)) << 16;
        const int64_t kblocks = p.k / 32;
        // part j of K-step ks of this row (zeros for a row past the matrix), or
        // the Q4_K / Q5_K min-term correction values of the steps past the weights
        auto part_values = [&](const U &u, bool live, const uint8_t *wrow, int ks, int j, uint32_t (&hi)[VW / 2],
                               uint32_t (&lo)[VW / 2]) {
#pragma unroll
            for (int w = 0; w < VW / 2; w++) { hi[w] = 0u; lo[w] = 0u; }
            if (!live) return;
            if (ks < KS_W) {
                if (H2) {
                    u.unpack_h2(ks, hi);
                } else {
                    float v[VW];
                    u.unpack_f32(ks, v);
                    if (PRECISE) pack_split<VW>(v, hi, lo);
                    else pack_single<VW>(v, hi);
                }
            } else if (WT == GGUF_Q4_K || WT == GGUF_Q5_K) {
                const int64_t nsb = p.k / 256;
                const int64_t sb0 = ((int64_t)ks * TG_BK - p.k) / 8;
                float v[VW];
#pragma unroll
                for (int e = 0; e < U::CHUNKS; e++) {
                    const int64_t sb = sb0 + U::chunk(j, e);
                    uint4 hdr = make_uint4(0, 0, 0, 0);
                    if (sb < nsb) hdr = *reinterpret_cast<const uint4 *>(wrow + sb * block_bytes(WT));
                    const uint32_t sc[3] = {hdr.y, hdr.z, hdr.w};
                    const float dmin = h2f(hdr.x >> 16);
#pragma unroll
                    for (int jj = 0; jj < 8; jj++) {
                        int sv, mv;
                        q4k_scale_min(sc, jj, sv, mv);
                        v[8 * e + jj] = sb < nsb ? __fmul_rn(dmin, (float)mv) : 0.0f;
                    }
                }
                pack_single<VW>(v, hi);
            }
        };
        // K-step ks (running index itk) of this row into its TMEM A stage
        auto produce_row = [&](const U (&uu)[PARTS], bool live, const uint8_t *wrow, int ks, int itk) -> bool {
            const int sa = itk % STA;
            const uint32_t pha = (uint32_t)(itk / STA) & 1u;
            // warp-uniform outcome: the TMEM stores below are warp-collective
            bool ok = !*abort_flag && tc::mbar_wait(&empty_a[sa], pha ^ 1u);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) { if (lane == 0) fail(4); return false; }
            tc::tc_fence_after();
            const uint32_t acol = tmem + tlane + (uint32_t)(S::A_COL0 + sa * 32 * S::OPS);
#pragma unroll
            for (int j = 0; j < PARTS; j++) {
                uint32_t hi[VW / 2], lo[VW / 2];
                part_values(uu[j], live, wrow, ks, j, hi, lo);
#pragma unroll
                for (int e = 0; e < U::CHUNKS; e++) {
                    const uint32_t c = acol + 4 * U::chunk(j, e);
                    tc::tmem_st_32x32b_x4(c, hi[4 * e], hi[4 * e + 1], hi[4 * e + 2], hi[4 * e + 3]);
                    if (PRECISE) tc::tmem_st_32x32b_x4(c + 32, lo[4 * e], lo[4 * e + 1], lo[4 * e + 2], lo[4 * e + 3]);
                }
            }
            tc::tmem_st_wait();
            tc::tc_fence_before();
            tc::mbar_arrive(&full_a[sa]);
            return true;
        };
        int it0 = 0, pc = 0;
        for (int t = blockIdx.x; t < tiles_total && !*abort_flag; t += gridDim.x) {
            const TgTile d = tg_tile<MODE, BN>(p, t, KS);
            // this thread's weight row (gate_up: rows 0..63 gate, 64..127 the matching up rows)
            int64_t row;
            bool live;
            if (MODE == TG_MOE_GATE_UP) {
                row = r < 64 ? d.row0 + r : p.n / 2 + d.row0 + (r - 64);
                live = (r < 64 ? d.row0 + r : d.row0 + (r - 64)) < p.n / 2;
            } else {
                row = d.row0 + r;
                live = row < p.n;
            }
            const uint8_t *wrow = p.w + (MODE == TG_DENSE ? 0 : (int64_t)d.e * p.expert_stride) + (live ? row : 0) * p.rb;
            const int kw1 = d.k1 < KS_W ? d.k1 : KS_W;
            const int kfirst = d.k0 + ((grp - it0) % TG_GROUPS + TG_GROUPS) % TG_GROUPS;
            bool ok = true;
            int ks = kfirst;
            if (p.pstages > 0) {
                const int PS = p.pstages;
                for (int c = d.k0 / p.pkc; c * p.pkc < kw1 && ok; c++, pc++) {
                    const int ps = pc % PS;
                    const int c1 = (c + 1) * p.pkc < kw1 ? (c + 1) * p.pkc : kw1;
                    ok = __all_sync(0xffffffffu, tc::mbar_wait(&pfull[ps], (uint32_t)(pc / PS) & 1u));
                    if (!ok) { if (lane == 0) fail(4); break; }
                    // the row in the buffer, offset so that the type's block
                    // arithmetic on a K-step lands in the buffer
                    const int64_t x0 = p.pchunked ? (int64_t)c * p.pb256 / 16 * 16 : 0;
                    const uint8_t *vrow = sP + (int64_t)ps * p.pstage_bytes + (int64_t)r * p.ppitch - x0;
                    for (; ks < c1 && ok; ks += TG_GROUPS) {
                        U uu[PARTS];
#pragma unroll
                        for (int j = 0; j < PARTS; j++)
                            if (live) uu[j].load(vrow, ks, j, kblocks);
                        ok = produce_row(uu, live, wrow, ks, it0 + ks - d.k0);
                    }
                    __syncwarp();   // every lane's reads of the buffer are done
                    if (lane == 0) tc::mbar_arrive(&pempty[ps]);
                }
            } else {
                // the next own K-step's bytes are loaded while this one is unpacked
                U un[PARTS];
                auto load_row = [&](U (&uu)[PARTS], int kk) {
                    if (kk >= kw1 || !live) return;
#pragma unroll
                    for (int j = 0; j < PARTS; j++) uu[j].load(wrow, kk, j, kblocks);
                };
                load_row(un, ks);
                for (; ks < kw1 && ok; ks += TG_GROUPS) {
                    U uu[PARTS];
#pragma unroll
                    for (int j = 0; j < PARTS; j++) uu[j] = un[j];
                    load_row(un, ks + TG_GROUPS);
                    ok = produce_row(uu, live, wrow, ks, it0 + ks - d.k0);
                }
            }
            // steps past the weights (correction columns)
            for (; ks < d.k1 && ok; ks += TG_GROUPS) {
                U uu[PARTS];
                ok = produce_row(uu, live, wrow, ks, it0 + ks - d.k0);
            }
            if (!ok) break;
            it0 += d.k1 - d.k0;
        }
      } else {
        // ================= A producers.  The 8 warps form TG_GROUPS groups;
        // group g builds the A tiles of the K-steps whose running index is g
        // modulo TG_GROUPS, so that several K-steps are unpacked at once.  In a
        // group, thread p takes part p % PARTS of tile rows p / PARTS + RP * i
        // (RP = threads per group / PARTS rows per pass).
        using U = KQ<WT>;
        constexpr int GW = (TG_PRODUCERS / 32) / TG_GROUPS;   // warps per group
        constexpr int PARTS = U::PARTS, RP = 32 * GW / PARTS, TPT = TG_BM / RP;
        constexpr int VW = 8 * U::CHUNKS;  // fp32 values per task
        // own K-steps loaded ahead from global memory (unstaged rows): the next
        // one, TG_GROUPS K-steps later in the stream
        constexpr int DEPTH = 1;
        // lane -> (row, part): each group of 8 lanes takes one part of 8
        // different rows, so a 16-byte swizzled store is conflict-free within
        // every 8-lane phase, and the parts of a row are in the same warp so a
        // warp-wide load still reads whole 32-byte sectors
        const int grp = (warp - 2) / GW, pw = (warp - 2) % GW, pl = lane;
        const int part = (pl >> 3) % PARTS;
        const int r0 = (32 / PARTS) * pw + (pl & 7) + 8 * (pl / (8 * PARTS));
        const int64_t kblocks = p.k / 32;
        // one task: unpack (weight steps) or the Q4_K / Q5_K min-term correction
        // values dmin * m_j of 8 sub-blocks per chunk (steps past the weights)
        auto task = [&](const U &u, bool live_i, const uint8_t *wrow_i, int ks, uint32_t (&hi)[VW / 2],
                        uint32_t (&lo)[VW / 2]) {
#pragma unroll
            for (int w = 0; w < VW / 2; w++) { hi[w] = 0u; lo[w] = 0u; }
            if (!live_i) return;
            if (ks < KS_W) {
                if (H2) {
                    u.unpack_h2(ks, hi);
                } else {
                    float v[VW];
                    u.unpack_f32(ks, v);
                    if (PRECISE) pack_split<VW>(v, hi, lo);
                    else pack_single<VW>(v, hi);
                }
            } else if (WT == GGUF_Q4_K || WT == GGUF_Q5_K) {
                // chunk c of this step holds the corrections of super-block
                // (ks * 64 - k) / 64 + c of the row
                const int64_t nsb = p.k / 256;
                const int64_t sb0 = ((int64_t)ks * TG_BK - p.k) / 8;
                float v[VW];
#pragma unroll
                for (int e = 0; e < U::CHUNKS; e++) {
                    const int64_t sb = sb0 + U::chunk(part, e);
                    uint4 hdr = make_uint4(0, 0, 0, 0);
                    if (sb < nsb) hdr = *reinterpret_cast<const uint4 *>(wrow_i + sb * block_bytes(WT));
                    const uint32_t sc[3] = {hdr.y, hdr.z, hdr.w};
                    const float dmin = h2f(hdr.x >> 16);
#pragma unroll
                    for (int jj = 0; jj < 8; jj++) {
                        int sv, mv;
                        q4k_scale_min(sc, jj, sv, mv);
                        v[8 * e + jj] = sb < nsb ? __fmul_rn(dmin, (float)mv) : 0.0f;
                    }
                }
                pack_single<VW>(v, hi);
            }
        };
        // K-step ks (running index itk): wait for its stage, then unpack and
        // store one task at a time (few live registers), signal the MMA
        auto produce = [&](const U (&uu)[TPT], const bool (&live)[TPT], const uint8_t *const (&wrow)[TPT], int ks,
                           int itk) -> bool {
            const int s = itk % STA;
            const uint32_t ph = (uint32_t)(itk / STA) & 1u;
            if (*abort_flag) return false;
            if (!tc::mbar_wait(&empty_a[s], ph ^ 1u)) { fail(4); return false; }
            uint8_t *tile = sA + s * S::A_STAGE;
#pragma unroll
            for (int i = 0; i < TPT; i++) {
                uint32_t hi[VW / 2], lo[VW / 2];
                task(uu[i], live[i], wrow[i], ks, hi, lo);
                store_sw128_task<U>(tile, r0 + RP * i, part, hi);
                if (PRECISE) store_sw128_task<U>(tile + TG_A_BYTES, r0 + RP * i, part, lo);
            }
            tc::fence_proxy_async_smem();
            tc::mbar_arrive(&full_a[s]);
            return true;
        };
        int it0 = 0;   // running index of the tile's first K-step
        int pc = 0;    // staged chunks consumed
        for (int t = blockIdx.x; t < tiles_total && !*abort_flag; t += gridDim.x) {
            const TgTile d = tg_tile<MODE, BN>(p, t, KS);
            bool live[TPT];
            const uint8_t *wrow[TPT];
            const uint8_t *wbase = p.w + (MODE == TG_DENSE ? 0 : (int64_t)d.e * p.expert_stride);
#pragma unroll
            for (int i = 0; i < TPT; i++) {
                const int r = r0 + RP * i;
                // gate_up tiles: rows 0..63 are gate rows, 64..127 the matching up rows
                int64_t row;
                if (MODE == TG_MOE_GATE_UP) {
                    row = r < 64 ? d.row0 + r : p.n / 2 + d.row0 + (r - 64);
                    live[i] = (r < 64 ? d.row0 + r : d.row0 + (r - 64)) < p.n / 2;
                } else {
                    row = d.row0 + r;
                    live[i] = row < p.n;
                }
                wrow[i] = wbase + (live[i] ? row : 0) * p.rb;
            }
            const int kw1 = d.k1 < KS_W ? d.k1 : KS_W;  // weight K steps of this tile
            // this group's first K-step of the tile
            const int kfirst = d.k0 + ((grp - it0) % TG_GROUPS + TG_GROUPS) % TG_GROUPS;
            bool ok = true;
            if (p.pstages > 0) {
                // staged: chunk c of the tile's weight steps waits in buffer pc % pstages
                const int PS = p.pstages;
                int ks = kfirst;
                for (int c = d.k0 / p.pkc; c * p.pkc < kw1 && ok; c++, pc++) {
                    const int ps = pc % PS;
                    const int c1 = (c + 1) * p.pkc < kw1 ? (c + 1) * p.pkc : kw1;
                    if (!tc::mbar_wait(&pfull[ps], (uint32_t)(pc / PS) & 1u)) { fail(4); ok = false; break; }
                    // row i of the buffer, offset so that the type's block
                    // arithmetic on a K-step of the row lands in the buffer
                    const int64_t x0 = p.pchunked ? (int64_t)c * p.pb256 / 16 * 16 : 0;
                    const uint8_t *buf = sP + (int64_t)ps * p.pstage_bytes;
                    const uint8_t *vrow[TPT];
#pragma unroll
                    for (int i = 0; i < TPT; i++) vrow[i] = buf + (int64_t)(r0 + RP * i) * p.ppitch - x0;
                    for (; ks < c1 && ok; ks += TG_GROUPS) {
                        U u[TPT];
#pragma unroll
                        for (int i = 0; i < TPT; i++)
                            if (live[i]) u[i].load(vrow[i], ks, part, kblocks);
                        ok = produce(u, live, wrow, ks, it0 + ks - d.k0);
                    }
                    __syncwarp();   // every lane's reads of the buffer are done
                    if (lane == 0) tc::mbar_arrive(&pempty[ps]);
                }
                // steps past the weights (correction columns)
                for (; ks < d.k1 && ok; ks += TG_GROUPS) {
                    U u[TPT];
                    ok = produce(u, live, wrow, ks, it0 + ks - d.k0);
                }
            } else {
                U u[DEPTH][TPT];   // tasks of this group's next DEPTH K-steps
                auto load_step = [&](U (&uu)[TPT], int ks) {
                    if (ks >= kw1) return;
#pragma unroll
                    for (int i = 0; i < TPT; i++)
                        if (live[i]) uu[i].load(wrow[i], ks, part, kblocks);
                };
#pragma unroll
                for (int dd = 0; dd < DEPTH; dd++) load_step(u[dd], kfirst + TG_GROUPS * dd);
                for (int ks = kfirst; ks < d.k1 && ok; ks += TG_GROUPS * DEPTH) {
#pragma unroll
                    for (int dd = 0; dd < DEPTH; dd++) {
                        const int kk = ks + TG_GROUPS * dd;
                        if (ok && kk < d.k1) {
                            ok = produce(u[dd], live, wrow, kk, it0 + kk - d.k0);
                            load_step(u[dd], kk + TG_GROUPS * DEPTH);   // DEPTH own K-steps ahead
                        }
                    }
                }
            }
            if (!ok) break;
            it0 += d.k1 - d.k0;
        }
      }
    } else if (warp < TG_LOADER_WARP) {
        // ================= epilogue
        const int q = warp & 3;
        int i = 0;
        int ochunk = 0;   // MoE down: bulk output stores issued (staging buffer ochunk & 1)
        for (int t = blockIdx.x; t < tiles_total; t += gridDim.x, i++) {
            const TgTile d = tg_tile<MODE, BN>(p, t, KS);
            const int b = i & 1;
            // MoE: the tile's route ids (and route weights), lane l holding routes
            // l, 32 + l, ...; loaded before the wait for the accumulator
            int rtv[MODE == TG_DENSE ? 1 : BN / 32];
            float wv[MODE == TG_DENSE ? 1 : BN / 32];
            if (MODE != TG_DENSE) {
#pragma unroll
                for (int c = 0; c < BN / 32; c++) {
                    const bool in = 32 * c + lane < d.n_eff;
                    rtv[c] = in ? p.route_list[d.route0 + 32 * c + lane] : 0;
                    wv[c] = (MODE == TG_MOE_DOWN && p.ysum && p.route_w && in) ? p.route_w[rtv[c]] : 1.0f;
                }
            }
            // warp-uniform outcome: the TMEM loads below are warp-collective
            const bool ok = __all_sync(0xffffffffu, tc::mbar_wait(&tfull[b], (uint32_t)(i >> 1) & 1u));
            if (!ok && lane == 0) fail(8);
            tc::tc_fence_after();
            const bool go = __all_sync(0xffffffffu, ok && !*abort_flag);
            if (MODE == TG_DENSE) {
                const int64_t orow = d.row0 + 32 * q + lane;
#pragma unroll 1
                for (int c = 0; c * 32 < BN && go; c++) {
                    uint32_t rr[32];
                    tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * BN + 32 * c), rr);
                    tc::tmem_ld_wait();
                    if (p.ystore) {
                        // this warp's 32 weight rows x 32 activation rows as one box:
                        // element (activation row jj, weight row lane) in the output
                        // dtype, then one bulk tensor store (edges past m, n clipped)
                        constexpr int ES = OT == GGUF_F32 ? 4 : 2;
                        uint8_t *ob = reinterpret_cast<uint8_t *>(xbuf) + (q * 2 + (ochunk & 1)) * (32 * 32 * ES);
                        if (lane == 0) tc::bulk_wait_read<1>();   // the box's previous store has read it
                        __syncwarp();
#pragma unroll
                        for (int jj = 0; jj < 32; jj++) {
                            const float v = __uint_as_float(rr[jj]);
                            if (OT == GGUF_F32) reinterpret_cast<float *>(ob)[jj * 32 + lane] = v;
                            else if (OT == GGUF_BF16) reinterpret_cast<uint16_t *>(ob)[jj * 32 + lane] = f2bf_rn(v);
                            else reinterpret_cast<uint16_t *>(ob)[jj * 32 + lane] = f2h_rn(v);
                        }
                        tc::fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) {
                            tc::tma_store_2d(&map_y, ob, (int32_t)(d.row0 + 32 * q), (int32_t)(d.m0 + 32 * c));
                            tc::bulk_commit();
                        }
                        ochunk++;
                        continue;
                    }
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
                // the chunk's rows leave through a staging buffer: bulk copies into z,
                // or bulk reduce-adds of the weighted rows into the token rows
                const bool staged = !p.ysum || p.ysum_bulk;
#pragma unroll
                for (int c = 0; c < BN / 32; c++) {
                    // the chunk count is the same in the 4 warps (they meet at named
                    // barriers); a warp whose wait failed skips the work only
                    if (c * 32 >= d.n_eff) break;
                    uint32_t rr[32];
                    const int rt_l = rtv[c];
                    const float w_l = wv[c];
                    const int rows = d.n_eff - 32 * c < 32 ? d.n_eff - 32 * c : 32;
                    float *ob = xbuf + (ochunk & 1) * (32 * 128);
                    if (staged) {
                        // the buffer's previous bulk copies have read it (each lane of
                        // warp 10 waits for its own)
                        if (warp == 10) tc::bulk_wait_read<1>();
                        tg_named_bar(2, 128);
                    }
                    if (go) {
                        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * BN + 32 * c), rr);
                        tc::tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int jj = 0; jj < 32; jj++) rr[jj] = 0u;
                    }
                    if (!staged) {
#pragma unroll
                        for (int jj = 0; jj < 32; jj++) {
                            if (go && jj < rows) {  // uniform within the warp
                                // fused weighted sum: w * (W_e . h_route) added into the
                                // token's fp32 row (the 32 lanes: 128 consecutive bytes)
                                const int rt = __shfl_sync(0xffffffffu, rt_l, jj);
                                const float wr = __shfl_sync(0xffffffffu, w_l, jj);
                                if (orow < p.n)
                                    atomicAdd(&p.ysum[(int64_t)(rt / p.top_k) * p.n + orow], wr * __uint_as_float(rr[jj]));
                            }
                        }
                    } else {
                        // the routes' output values in 128-column blocks, routes at their
                        // grouped positions: the chunk's rows of this column block are one
                        // contiguous run, written by one bulk copy from the staging buffer
#pragma unroll
                        for (int jj = 0; jj < 32; jj++) {
                            const float wr = __shfl_sync(0xffffffffu, w_l, jj);   // 1 without ysum
                            ob[jj * 128 + 32 * q + lane] = wr * __uint_as_float(rr[jj]);
                        }
                        tc::fence_proxy_async_smem();
                        tg_named_bar(2, 128);
                        if (warp == 10 && go) {
                            if (p.ysum) {
                                // lane l adds route row l (weighted) into its token's row:
                                // the tile's columns, clipped at n
                                if (lane < rows) {
                                    const int64_t cols = p.n - d.row0 < 128 ? p.n - d.row0 : 128;
                                    tc::bulk_reduce_add_f32(p.ysum + (int64_t)(rt_l / p.top_k) * p.n + d.row0,
                                                            ob + lane * 128, (uint32_t)cols * 4u);
                                }
                                tc::bulk_commit();
                            } else if (lane == 0) {
                                float *dst = p.yacc + (((int64_t)(d.row0 >> 7) * p.zrows + d.route0 + 32 * c) << 7);
                                tc::bulk_store(dst, ob, (uint32_t)rows * 512u);
                                tc::bulk_commit();
                            }
                        }
                        ochunk++;
                    }
                }
            } else {
                // gate rows in TMEM lanes 0..63 (q = 0, 1), up rows in 64..127 (q = 2, 3).
                // Per chunk of 32 routes: all four warps park their values in
                // xbuf[gate/up][route][i], then warp q finishes routes q, q+4, ...:
                // lane l takes h columns i = l and 32 + l, one q8_1 block each.
                const int64_t idim = p.n / 2;
                const int64_t hrb = idim / 32 * Q8_1_BYTES;
                float *xg = xbuf, *xu = xbuf + 32 * 64;
#pragma unroll 1
                for (int c = 0; c * 32 < BN; c++) {
                    const bool any = go && 32 * c < d.n_eff;  // uniform across the 4 warps
                    if (any) {
                        uint32_t rr[32];
                        tc::tmem_ld_32x32b_x32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * BN + 32 * c), rr);
                        tc::tmem_ld_wait();
                        float *dst = (q < 2 ? xg : xu) + 32 * (q & 1) + lane;
#pragma unroll
                        for (int jj = 0; jj < 32; jj++) dst[jj * 64] = __uint_as_float(rr[jj]);
                    }
                    tg_named_bar(1, 128);
                    if (any) {
                        // this chunk's route ids (a register array indexed by the loop count)
                        int rt_l = rtv[0];
#pragma unroll
                        for (int cc = 1; cc < BN / 32; cc++)
                            if (c == cc) rt_l = rtv[cc];
#pragma unroll 4
                        for (int jj = q; jj < 32; jj += 4) {
                            const int j = 32 * c + jj;
                            if (j >= d.n_eff) break;  // uniform within the warp
                            const int64_t rt = __shfl_sync(0xffffffffu, rt_l, jj);
#pragma unroll
                            for (int hb = 0; hb < 2; hb++) {
                                const int il = 32 * hb + lane;
                                const int64_t icol = d.row0 + il;  // column of h
                                const float gv = xg[jj * 64 + il], uv = xu[jj * 64 + il];
                                // silu in fp32 with the fast exponential and division (a few ulp of
                                // fp32, far below the bf16 rounding of h that follows)
                                const float hf = __fdividef(gv, 1.0f + __expf(-gv)) * uv;
                                const uint16_t hbits = f2bf_rn(hf);
                                const float hx = bf2f(hbits);  // the intermediate in the activation dtype
                                if (p.hbf) p.hbf[rt * idim + icol] = hbits;
                                // q8_1 of the 32 columns of this warp: amax on the (non-negative) float bits
                                const float amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hx))));
                                const float dq = __fdiv_rn(amax, 127.0f);
                                const int qv = dq != 0.0f ? (int)roundf(__fdiv_rn(hx, dq)) : 0;
                                const int sum = __reduce_add_sync(0xffffffffu, qv);
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
                                    // the fused down GEMM's operand: rows in grouped order
                                    const int64_t hr = p.h16_grouped ? (int64_t)d.route0 + j : rt;
                                    const float v = h2f(dh) * (float)qv;
                                    const uint16_t vh = f2h_rn(v);
                                    p.h16[hr * p.hpitch + icol] = vh;
                                    if (p.h16lo) p.h16lo[hr * p.hpitch + icol] = f2h_rn(v - h2f(vh));
                                    if (p.hpitch > idim) {
                                        // min-term correction column of this q8_1 block (Q4_K / Q5_K down
                                        // weights), and the zero padding of the row (written once,
                                        // by the first column tile)
                                        if (lane == 0) {
                                            const uint16_t sh = f2h_rn(__fmul_rn(dq, (float)sum));
                                            p.h16[hr * p.hpitch + idim + icol / 32] = f2h_rn(h2f(dh) * (float)sum - h2f(sh));
                                            if (p.h16lo) p.h16lo[hr * p.hpitch + idim + icol / 32] = 0;
                                        }
                                        if (d.row0 == 0 && hb == 0)
                                            for (int64_t c2 = idim + idim / 32 + lane; c2 < p.hpitch; c2 += 32) {
                                                p.h16[hr * p.hpitch + c2] = 0;
                                                if (p.h16lo) p.h16lo[hr * p.hpitch + c2] = 0;
                                            }
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
        // bulk output copies finish before the CTA's shared memory is released
        // (each lane waits for the groups it committed)
        tc::bulk_wait_all();
    } else if (lane == 0 && p.pstages > 0) {
        // ================= packed-weight loader: chunk c of a tile (K-steps
        // [c * pkc, (c + 1) * pkc) of its weight steps) into buffer pc % pstages:
        // the 16-byte-aligned window of the chunk's bytes of 128 rows (64 gate
        // + 64 up rows for gate_up), or whole rows
        const int PS = p.pstages;
        int pc = 0, last = 0;
        bool ok = true;
        for (int t = blockIdx.x; t < tiles_total && ok && !*abort_flag; t += gridDim.x) {
            const TgTile d = tg_tile<MODE, BN>(p, t, KS);
            const int kw1 = d.k1 < KS_W ? d.k1 : KS_W;
            const int32_t z = MODE == TG_DENSE ? 0 : d.e;
            for (int c = d.k0 / p.pkc; c * p.pkc < kw1; c++, pc++) {
                const int ps = pc % PS;
                if (*abort_flag) { ok = false; break; }
                if (!tc::mbar_wait(&pempty[ps], ((uint32_t)(pc / PS) & 1u) ^ 1u)) { fail(32); ok = false; break; }
                tc::mbar_arrive_expect_tx(&pfull[ps], (uint32_t)(TG_BM * p.ppitch));
                uint8_t *dst = sP + (int64_t)ps * p.pstage_bytes;
                // x in 8-byte elements of the tensor map
                const int32_t x = p.pchunked ? (int32_t)((int64_t)c * p.pb256 / 16 * 2) : 0;
                if (MODE == TG_MOE_GATE_UP) {
                    tc::tma_load_3d(dst, &map_w, &pfull[ps], x, (int32_t)(d.row0 / p.pgroup), z);
                    tc::tma_load_3d(dst + 64 * p.ppitch, &map_w, &pfull[ps], x,
                                    (int32_t)((p.n / 2 + d.row0) / p.pgroup), z);
                } else {
                    tc::tma_load_3d(dst, &map_w, &pfull[ps], x, (int32_t)(d.row0 / p.pgroup), z);
                }
                last = pc + 1;
            }
        }
        if (*abort_flag)  // copies already issued land before the CTA exits
            for (int i = last - PS < 0 ? 0 : last - PS; i < last; i++)
                tc::mbar_wait(&pfull[i % PS], (uint32_t)(i / PS) & 1u);
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

// the output y[m][ldy] (element type ot) as a 2-D tensor map with 32 x 32
// boxes, for the dense epilogue's bulk tensor stores; false when its base or
// row stride is not 16-byte aligned
inline bool tg_make_out_map(CUtensorMap *map, void *y, int ot, int64_t n, int64_t m, int64_t ldy) {
    auto enc = tensor_map_encoder();
    const int64_t es = ot == GGUF_F32 ? 4 : 2;
    if (!enc || (reinterpret_cast<uintptr_t>(y) & 15) || (ldy * es) % 16 || n <= 0 || m <= 0) return false;
    cuuint64_t gdim[2] = {(cuuint64_t)n, (cuuint64_t)m};
    cuuint64_t gstride[1] = {(cuuint64_t)(ldy * es)};
    cuuint32_t box[2] = {32, 32};
    cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt = ot == GGUF_F32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                   : ot == GGUF_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(map, dt, 2, y, gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
               CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Staging of the packed weight rows (sets the p.p* fields and the tensor map;
// p.pstages = 0 when the rows cannot be staged, and the producers then load
// from global memory).  The weights are E matrices of `rows` rows of k values,
// expert_stride bytes apart (E = 1: one matrix); a buffer holds 128 rows,
// taken as boxes of box_rows rows.  base_bytes: shared memory the kernel uses
// before the ring.
//   chunked : row bytes a multiple of 16 and k a multiple of 256; a buffer is
//             the 16-byte-aligned window over one 256-value chunk of the rows;
//   rows    : otherwise, whole rows, taken g at a time so that a line of the
//             tensor map is a multiple of 16 bytes (g * row bytes <= 2048).
inline void tg_plan_staging(TgParams &p, CUtensorMap *map, int wt, const uint8_t *w, int64_t rows, int64_t E,
                            int64_t expert_stride, int64_t k, int box_rows, int base_bytes) {
    p.pstages = 0;
    p.pkc = 1;
    p.pgroup = 1;
    auto enc = tensor_map_encoder();
    const int64_t rb = k / block_elems(wt) * block_bytes(wt);
    const int ksw = (int)((k + TG_BK - 1) / TG_BK);
    if (!enc || rb <= 0 || (reinterpret_cast<uintptr_t>(w) & 15) || (E > 1 && expert_stride % 16)) return;
    int g = 1, chunked = 0;
    int64_t pitch = 0;
    if (rb % 16 == 0 && k % 256 == 0 && tg_chunk_pitch(wt) > 0) {
        chunked = 1;
        pitch = tg_chunk_pitch(wt);
    } else {
        while ((g * rb) % 16) g *= 2;
        if (g > 16 || rows % g || box_rows % g || g * rb > 2048) return;
        pitch = rb;
    }
    // a box that fills part of a buffer (gate_up: 64 gate rows, then 64 up rows)
    // must leave the next box 128-byte aligned
    if (box_rows < TG_BM && (box_rows * pitch) % 128) return;
    const int64_t stage = (TG_BM * pitch + 1023) / 1024 * 1024;
    int64_t ps = (TG_SMEM_MAX - base_bytes) / stage;
    if (ps > TG_MAX_PSTAGES) ps = TG_MAX_PSTAGES;
    if (ps < 2) return;
    const int64_t line = chunked ? rb : g * rb;   // bytes of one line of the map
    cuuint64_t gdim[3] = {(cuuint64_t)(line / 8), (cuuint64_t)(rows / g), (cuuint64_t)E};
    cuuint64_t gstride[2] = {(cuuint64_t)line, (cuuint64_t)(E > 1 ? expert_stride : rows * rb)};
    cuuint32_t box[3] = {(cuuint32_t)((chunked ? pitch : line) / 8), (cuuint32_t)(box_rows / g), 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT64, 3, const_cast<uint8_t *>(w), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return;
    p.pstages = (int)ps;
    p.pkc = chunked ? 4 : ksw;
    p.pchunked = chunked;
    p.pgroup = g;
    p.ppitch = pitch;
    p.pstage_bytes = stage;
    p.pb256 = tg_chunk_bytes(wt);
}

template <int WT, int BN, bool PRECISE, int MODE, int OT>
inline cudaError_t tg_launch(const CUtensorMap &mh, const CUtensorMap &ml, const CUtensorMap &mw, const CUtensorMap &my,
                             const TgParams &p, int grid, cudaStream_t s) {
    using S = TgShape<WT, BN, PRECISE, MODE>;
    auto kern = tg_kernel<WT, BN, PRECISE, MODE, OT>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, TG_SMEM_MAX);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    int *err = tg_error_word();
    if (!err) return cudaErrorInvalidSymbol;
    const int64_t smem = S::BASE + (int64_t)p.pstages * p.pstage_bytes;
    if (smem > TG_SMEM_MAX) return cudaErrorInvalidValue;
    kern<<<grid, TG_THREADS, (size_t)smem, s>>>(mh, ml, mw, my, p, err);
    return cudaGetLastError();
}

template <int WT, int BN, bool PRECISE, int MODE>
constexpr int tg_base_bytes() {
    return TgShape<WT, BN, PRECISE, MODE>::BASE;
}

}  // namespace gg
