// Tensor-core MMVQ for 5..8 tokens of Q6_K rows: the per-group integer dot
// products of the blockwise formula run on warp-level int8 MMAs
// (mma.sync m16n8k16 u8 x s8 -> s32).  One MMA is one 16-value scale group of
// 16 weight rows against 8 tokens, so its s32 accumulator is exactly
// sum_i q6_i * q_a,i over the group (q6 in 0..63, stored unsigned); the -32
// offset of the Q6_K values is removed exactly with the group's activation sum
// (32 * sum_i q_a,i, precomputed per token):
//   y = d * sum_b d_a,b * sum_{j in b} sc_j * (S_j - 32 Q_j)
// where b runs over the q8_1 blocks (two scale groups each).  The sc_j products
// are summed in int32 per q8_1 block, so each block costs one int -> float
// conversion per output; d and d_a are applied in fp32.
//
// Work split as in the Q4_K kernel: a CTA of NW warps owns 16-row tiles, warp w
// takes super-blocks [w * nsb / NW, (w + 1) * nsb / NW) of every tile, and the
// warps' partial results of up to 4 tiles are summed in a fixed order.
// Weights: Q6_K super-blocks (210 bytes) are only 2-byte aligned, so lane l
// loads the 16-byte-aligned cover of row l % 16 of the item, chunks
// l / 16 + 2 i (one 16-byte load each; 14 chunks cover any 210-byte span),
// into registers one item ahead; the chunks go to the warp's shared buffer,
// where each lane reads its words with a funnel shift when the row is
// 2 mod 4 aligned.  The last row of a weight view never reads past its end
// (2-byte loads for the bytes of its last chunk).
#pragma once

#include "mmvq_mma.cuh"

namespace gg {

__device__ __forceinline__ void mma_16816_u8s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t b0) {
    asm("mma.sync.aligned.m16n8k16.row.col.s32.u8.s8.s32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%7,%7,%7,%7};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(b0), "r"(0));
}

// the 4 bytes at a 2-byte-aligned shared-memory address
__device__ __forceinline__ uint32_t lds_w_a2(const uint8_t *p) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t *b = reinterpret_cast<const uint32_t *>(a & ~uintptr_t(3));
    return __funnelshift_r(b[0], b[1], (a & 2) ? 16 : 0);
}

constexpr int Q6_ROW_PITCH = 224;                 // 14 chunks: the cover of any 210-byte span
constexpr int Q6_WST = 16 * Q6_ROW_PITCH + 16;    // one warp's buffer (+ a word read past the last row)

struct Q6Smem {
    int64_t xs, xs_pitch, da, qs, red, wst, total;
};
__host__ __device__ inline Q6Smem q6_smem_layout(int64_t k, int nw, int grp, int nt) {
    const int64_t nblk = k / 32, ngr = k / 16, tok = 8 * (int64_t)nt;
    Q6Smem L;
    L.xs = 0;                                               // 8*nt token rows of nblk x 32 quants (+8 B pad)
    L.xs_pitch = (nblk * 40 + 127) / 128 * 128 + 32;        // 40 B per block; pitch = 32 mod 128 bytes
    L.da = L.xs + tok * L.xs_pitch;                         // float [nblk][8*nt]: d_a
    L.qs = L.da + nblk * tok * 4;                           // int [ngr][8*nt]: 32 * sum of the group's quants
    L.red = L.qs + ngr * tok * 4;                           // float4 [2][grp][nw][nt][32]
    L.wst = L.red + 2 * (int64_t)grp * nw * nt * 32 * 16;   // [nw][Q6_WST] weight buffers
    L.total = L.wst + (int64_t)nw * Q6_WST;
    return L;
}

struct Q6Raw {
    uint4 c[7];      // chunks h + 2 i of this lane's row cover (h = lane / 16)
    uint32_t head;   // byte offset of the super-block in its cover
};

template <int NT>
__global__ void __launch_bounds__(256, 2)
    mmvq_mma_q6k_kernel(const MmvqSegs sg, int64_t k, int64_t rb, const uint8_t *__restrict__ xq, int m_act, int yt,
                        int grp) {
    constexpr int TOK = 8 * NT;
    const int64_t n = sg.rows();
    extern __shared__ __align__(16) uint8_t smem[];
    const int nw = blockDim.x >> 5;
    const Q6Smem L = q6_smem_layout(k, nw, grp, NT);
    uint8_t *xs = smem + L.xs;
    float *da = reinterpret_cast<float *>(smem + L.da);
    int *qs = reinterpret_cast<int *>(smem + L.qs);
    float4 *red = reinterpret_cast<float4 *>(smem + L.red);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nblk = (int)(k / 32), nsb = (int)(k / 256);
    const int64_t xrb = (int64_t)nblk * Q8_1_BYTES;
    const int pitch = (int)L.xs_pitch;
    const int64_t n_tiles = (n + 15) / 16;
    const int sb_lo = warp * nsb / nw, sb_hi = (warp + 1) * nsb / nw;
    uint8_t *wst = smem + L.wst + (int64_t)warp * Q6_WST;

    // ---- loads: lane l takes row rl = l % 16 of the tile, chunks ch + 2 i
    const int rl = lane & 15, ch = lane >> 4;
    int64_t cached_tile = -1;
    const uint8_t *rowp = nullptr;   // this lane's weight row (null past the view)
    bool row_last = false;           // the last row of its weight view
    auto load_item = [&](Q6Raw &R, int64_t tile, int sb) {
        if (tile != cached_tile) {
            const int64_t row = tile * 16 + rl;
            rowp = nullptr;
            row_last = false;
            if (row < n) {
                const int s = seg_index(sg, row);
                rowp = sg.w[s] + (row - (s ? sg.end[s - 1] : 0)) * rb;
                row_last = row + 1 == (sg.end[s] < n ? sg.end[s] : n);
            }
            cached_tile = tile;
        }
        R.head = 0;
        if (rowp == nullptr) return;
        const uint8_t *a = rowp + (int64_t)sb * Q6_K_BYTES;
        const uint32_t head = (uint32_t)(reinterpret_cast<uintptr_t>(a) & 15);
        const uint8_t *cover = a - head;
        const uint32_t end = head + Q6_K_BYTES;   // bytes of the cover that belong to the span
        const bool guard = row_last && sb == nsb - 1;
        R.head = head;
#pragma unroll
        for (int i = 0; i < 7; i++) {
            const uint32_t q = (uint32_t)(ch + 2 * i);
            if (16 * q >= end) continue;
            if (!guard || 16 * q + 16 <= end) {
                R.c[i] = __ldg(reinterpret_cast<const uint4 *>(cover + 16 * q));
            } else {   // the view's last bytes: 2-byte loads up to the span end
                uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
                for (int j = 0; j < 8; j++)
                    if (16 * q + 2 * j < end) w[j >> 1] |= (uint32_t)ld_u16(cover + 16 * q + 2 * j) << (16 * (j & 1));
                R.c[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
        }
    };

    // the first item's weights are requested before waiting for the kernel
    // that wrote the activations
    int64_t tile = blockIdx.x;
    Q6Raw wa, wb;
    if (sb_lo < sb_hi && tile < n_tiles) load_item(wa, tile, sb_lo);
    mmvq_pdl_enter(sg.chain);

    // ---- q8_1 rows into shared memory (quants of block b at b * 40 + 8),
    // d_a per block and 32 * (sum of the quants) per 16-value group
    for (int i = tid; i < TOK * nblk; i += blockDim.x) {
        const int tok = i / nblk, b = i - tok * nblk;
        uint32_t *dst = reinterpret_cast<uint32_t *>(xs + tok * pitch + b * 40 + 8);
        if (tok < m_act) {
            const uint32_t *src = reinterpret_cast<const uint32_t *>(xq + tok * xrb + (int64_t)b * Q8_1_BYTES + 4);
            int s0 = 0, s1 = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) {
                const uint32_t v = src[j];
                dst[j] = v;
                if (j < 4) s0 = __dp4a((int)v, 0x01010101, s0);
                else s1 = __dp4a((int)v, 0x01010101, s1);
            }
            qs[(2 * b) * TOK + tok] = 32 * s0;
            qs[(2 * b + 1) * TOK + tok] = 32 * s1;
        } else {
#pragma unroll
            for (int j = 0; j < 8; j++) dst[j] = 0u;
            qs[(2 * b) * TOK + tok] = 0;
            qs[(2 * b + 1) * TOK + tok] = 0;
        }
    }
    for (int i = tid; i < nblk * TOK; i += blockDim.x) {
        const int b = i / TOK, tok = i % TOK;
        da[i] = tok < m_act ? h2f(ld_u16(xq + tok * xrb + (int64_t)b * Q8_1_BYTES)) : 0.0f;
    }
    __syncthreads();

    const uint8_t *xg = xs + g * pitch + 8 + 4 * t;   // this lane's B word: token 8nt + g, values 4t .. 4t+3 of a group

    // one (tile, super-block) item; partial sums of rows g, g+8 x tokens 8nt + 2t, +1 into acc[nt]
    auto process = [&](const Q6Raw &R, int sb, float (&acc)[NT][4]) {
        // the item's 16 row covers into the warp's buffer
#pragma unroll
        for (int i = 0; i < 7; i++) {
            const int q = ch + 2 * i;
            if (16 * q < (int)R.head + Q6_K_BYTES)
                *reinterpret_cast<uint4 *>(wst + rl * Q6_ROW_PITCH + 16 * q) = R.c[i];
        }
        const uint32_t head0 = __shfl_sync(0xffffffffu, R.head, g), head1 = __shfl_sync(0xffffffffu, R.head, g + 8);
        __syncwarp();
        const uint8_t *b0 = wst + g * Q6_ROW_PITCH + head0, *b1 = wst + (g + 8) * Q6_ROW_PITCH + head1;
        const float d0 = h2f(*reinterpret_cast<const uint16_t *>(b0 + 208));
        const float d1 = h2f(*reinterpret_cast<const uint16_t *>(b1 + 208));
        uint32_t sc0[4], sc1[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            sc0[i] = lds_w_a2(b0 + 192 + 4 * i);
            sc1[i] = lds_w_a2(b1 + 192 + 4 * i);
        }
        uint32_t wl[2][2][2][2], wh[2][2][2];   // [row][h][ql half][s], [row][h][s]
#pragma unroll
        for (int h = 0; h < 2; h++)
#pragma unroll
            for (int s = 0; s < 2; s++) {
                wl[0][h][0][s] = lds_w_a2(b0 + 64 * h + 16 * s + 4 * t);
                wl[0][h][1][s] = lds_w_a2(b0 + 64 * h + 32 + 16 * s + 4 * t);
                wh[0][h][s] = lds_w_a2(b0 + 128 + 32 * h + 16 * s + 4 * t);
                wl[1][h][0][s] = lds_w_a2(b1 + 64 * h + 16 * s + 4 * t);
                wl[1][h][1][s] = lds_w_a2(b1 + 64 * h + 32 + 16 * s + 4 * t);
                wh[1][h][s] = lds_w_a2(b1 + 128 + 32 * h + 16 * s + 4 * t);
            }
        __syncwarp();   // every lane has its words before the buffer is rewritten
        float u[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int i = 0; i < 4; i++) u[nt][i] = 0.0f;
#pragma unroll
        for (int h = 0; h < 2; h++) {
#pragma unroll
            for (int q = 0; q < 4; q++) {
                // q8_1 block b = 8 sb + 4 h + q holds scale groups j = 2b, 2b + 1 (s = 0, 1):
                // values 128 h + 32 q + 16 s + 4 t + i of the super-block
                const int blk = sb * 8 + 4 * h + q;
                const int sh = 4 * (q >> 1);
                int T[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; nt++)
#pragma unroll
                    for (int i = 0; i < 4; i++) T[nt][i] = 0;
#pragma unroll
                for (int s = 0; s < 2; s++) {
                    const int j = 8 * h + 2 * q + s;   // scale group in the super-block
                    const uint32_t a0 = ((wl[0][h][q & 1][s] >> sh) & 0x0F0F0F0Fu) |
                                        (((wh[0][h][s] >> (2 * q)) & 0x03030303u) << 4);
                    const uint32_t a1 = ((wl[1][h][q & 1][s] >> sh) & 0x0F0F0F0Fu) |
                                        (((wh[1][h][s] >> (2 * q)) & 0x03030303u) << 4);
                    const int s0 = (int)(int8_t)(sc0[j >> 2] >> (8 * (j & 3)));
                    const int s1 = (int)(int8_t)(sc1[j >> 2] >> (8 * (j & 3)));
#pragma unroll
                    for (int nt = 0; nt < NT; nt++) {
                        const uint32_t bw = *reinterpret_cast<const uint32_t *>(xg + 8 * nt * pitch + blk * 40 + 16 * s);
                        int S[4];
                        mma_16816_u8s8(S, a0, a1, bw);
                        const int2 qq = *reinterpret_cast<const int2 *>(qs + (sb * 16 + j) * TOK + 8 * nt + 2 * t);
                        // accumulator i: row g (i < 2) or g+8, token 8nt + 2t + (i & 1)
                        T[nt][0] += s0 * (S[0] - qq.x);
                        T[nt][1] += s0 * (S[1] - qq.y);
                        T[nt][2] += s1 * (S[2] - qq.x);
                        T[nt][3] += s1 * (S[3] - qq.y);
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; nt++) {
                    const float2 dd = *reinterpret_cast<const float2 *>(da + blk * TOK + 8 * nt + 2 * t);
                    u[nt][0] = fmaf(dd.x, (float)T[nt][0], u[nt][0]);
                    u[nt][1] = fmaf(dd.y, (float)T[nt][1], u[nt][1]);
                    u[nt][2] = fmaf(dd.x, (float)T[nt][2], u[nt][2]);
                    u[nt][3] = fmaf(dd.y, (float)T[nt][3], u[nt][3]);
                }
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            acc[nt][0] = fmaf(d0, u[nt][0], acc[nt][0]);
            acc[nt][1] = fmaf(d0, u[nt][1], acc[nt][1]);
            acc[nt][2] = fmaf(d1, u[nt][2], acc[nt][2]);
            acc[nt][3] = fmaf(d1, u[nt][3], acc[nt][3]);
        }
    };

    int buf = 0, gi = 0;   // gi: tiles held in the current group
    for (; tile < n_tiles; tile += gridDim.x) {
        float acc[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int i = 0; i < 4; i++) acc[nt][i] = 0.0f;
        // items of this tile, two register sets in turn; the item after the
        // last one of the tile is the first of the next tile
        for (int sb = sb_lo; sb < sb_hi; sb += 2) {
            {
                const bool more = sb + 1 < sb_hi;
                const int64_t nt = more ? tile : tile + gridDim.x;
                if (nt < n_tiles) load_item(wb, nt, more ? sb + 1 : sb_lo);
            }
            process(wa, sb, acc);
            if (sb + 1 >= sb_hi) {
                wa = wb;   // odd count: the next tile's first item is in wb
                break;
            }
            {
                const bool more = sb + 2 < sb_hi;
                const int64_t nt = more ? tile : tile + gridDim.x;
                if (nt < n_tiles) load_item(wa, nt, more ? sb + 2 : sb_lo);
            }
            process(wb, sb + 1, acc);
        }
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
            red[(((buf * grp + gi) * nw + warp) * NT + nt) * 32 + lane] =
                make_float4(acc[nt][0], acc[nt][1], acc[nt][2], acc[nt][3]);
        gi++;
        // every `grp` tiles (and after the last), sum the warps' partial results
        // of the group's tiles in a fixed order
        if (gi == grp || tile + gridDim.x >= n_tiles) {
            __syncthreads();
            for (int i = tid; i < gi * 128 * NT; i += blockDim.x) {   // per tile: 16 rows x 8*NT tokens
                const int tt = i / (128 * NT), rem = i % (128 * NT), nt = rem >> 7, l = (rem >> 2) & 31, e = rem & 3;
                float s = 0.0f;
                for (int wj = 0; wj < nw; wj++) {
                    const float4 v = red[(((buf * grp + tt) * nw + wj) * NT + nt) * 32 + l];
                    s += e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
                }
                const int64_t t_of = tile - (int64_t)(gi - 1 - tt) * gridDim.x;
                const int64_t row = t_of * 16 + (l >> 2) + 8 * (e >> 1);
                const int tok = 8 * nt + 2 * (l & 3) + (e & 1);
                if (row < n && tok < m_act) seg_store(sg, yt, tok, row, s);
            }
            buf ^= 1;
            gi = 0;
        }
    }
}

inline int mma_q6k_warps(int64_t k) {
    int nw = (int)(k / 256 / 2);
    return nw < 1 ? 1 : nw > 8 ? 8 : nw;
}
// tiles per reduction group: the largest of 4, 2, 1 that leaves room for two
// CTAs per SM, else the largest that fits one (0: does not fit)
inline int mma_q6k_group(int64_t k, int nt) {
    const int64_t cap = (int64_t)device_info().smem_optin;
    for (int grp = 4; grp >= 1; grp /= 2)
        if (2 * (q6_smem_layout(k, mma_q6k_warps(k), grp, nt).total + 1024) <= cap) return grp;
    for (int grp = 4; grp >= 1; grp /= 2)
        if (q6_smem_layout(k, mma_q6k_warps(k), grp, nt).total <= cap) return grp;
    return 0;
}
inline bool mma_q6k_fits(int64_t k, int64_t m) { return m <= 8 && mma_q6k_group(k, 1) > 0; }

inline cudaError_t launch_mmvq_mma_q6k(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt,
                                       cudaStream_t s) {
    const int64_t n = sg.rows();
    const int nw = mma_q6k_warps(k), grp = mma_q6k_group(k, 1);
    if (grp == 0) return cudaErrorInvalidValue;
    const Q6Smem L = q6_smem_layout(k, nw, grp, 1);
    auto kern = mmvq_mma_q6k_kernel<1>;
    cudaError_t e = cudaSuccess;
    const int per_sm = kernel_occupancy(reinterpret_cast<const void *>(kern), nw * 32, (size_t)L.total, &e);
    if (per_sm == 0) return e;
    const int64_t n_tiles = (n + 15) / 16;
    int64_t grid = (int64_t)device_info().sm_count * per_sm;
    if (grid > n_tiles) grid = n_tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)(nw * 32));
    cfg.dynamicSmemBytes = (size_t)L.total;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, sg, k, k / 256 * (int64_t)Q6_K_BYTES, xq, (int)m, yt, grp);
}

}  // namespace gg
