// Tensor-core MMVQ for 5..32 tokens (Q4_K and Q5_K weights): the per-block int32 dot
// products of the blockwise formula run on warp-level int8 MMAs
// (mma.sync m16n8k32 s8 x s8 -> s32).  One MMA is one 32-value block of 16
// weight rows against 8 tokens (one n-tile; 2 or 4 n-tiles share the weight
// fragments for 9..32 tokens), so its s32 accumulator is exactly the block
// dot S_j of each (row, token) pair; scales are then applied per block in
// fp32 as in the dp4a kernel:
//   y += d * sum_j s_j * d_a,j * S_j  -  dmin * sum_j m_j * s_a,j
// At 8 tokens the dp4a form needs 16 dp4a per token per 64 weights, which
// GB300's int8 rate cannot issue as fast as HBM delivers the weights; here the
// operands need one LOP3 per 4 weights (Q4_K nibbles are non-negative int8)
// and the q8_1 quants are the B fragments as they are.  Q5_K adds the fifth
// bit of each quant from its 32 high-bit bytes (bit 2c of byte i for value i
// of sub-block 2c, bit 2c + 1 for sub-block 2c + 1): the quants stay
// non-negative int8 (0..31), so the same MMA and scale arithmetic apply.
// The min term of a super-block is one fp16 MMA: A = the rows' 8 six-bit
// mins, B = the 8 blocks' stored fp16 s_a (products exact in fp32).
//
// Work split.  A CTA of NW warps owns 16-row tiles; warp w takes super-blocks
// [w * nsb / NW, (w + 1) * nsb / NW) of every tile; the warps' partial results
// of up to 4 tiles are kept in shared memory and then summed in a fixed order
// (deterministic; one CTA barrier per group of tiles).
// The q8_1 rows (8 tokens) are copied once per CTA into shared memory with the
// 32 quants of each block on an 8-byte boundary; the weights of the next
// (tile, super-block) item load into registers while the current one computes.
#pragma once

#include "mmvq.cuh"

namespace gg {

__device__ __forceinline__ void mma_16832_s8(int (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(0));
}

__device__ __forceinline__ void mma_16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f));
}

// Shared-memory layout (bytes) for rows of nblk = K/32 q8_1 blocks; the
// warps' partial sums of up to `grp` tiles are kept before one reduction.
struct MmaSmem {
    int64_t xs, xs_pitch, da, saf, red, hdr, total;
};
__host__ __device__ inline MmaSmem mma_smem_layout(int64_t k, int nw, int grp, int nt) {
    const int64_t nblk = k / 32, nsb = k / 256, tok = 8 * (int64_t)nt;
    MmaSmem L;
    L.xs = 0;                                               // 8*nt token rows of nblk x 32 quants (+8 B pad)
    L.xs_pitch = (nblk * 40 + 127) / 128 * 128 + 32;        // 40 B per block; pitch = 32 mod 128 bytes
    L.da = L.xs + tok * L.xs_pitch;                         // float [nblk][8*nt]: d_a
    L.saf = L.da + nblk * tok * 4;                          // uint32 [nsb][nt][32]: s_a pairs for the min MMA
    L.red = L.saf + nsb * nt * 32 * 4;                      // float4 [2][grp][nw][nt][32]
    L.hdr = L.red;                                          // uint32 [8*nt][nblk] block headers while staging
    const int64_t red_end = L.red + 2 * (int64_t)grp * nw * nt * 32 * 16, hdr_end = L.hdr + tok * nblk * 4;
    L.total = red_end > hdr_end ? red_end : hdr_end;
    return L;
}

struct MmaWBase {
    uint4 h0, h1;        // headers of rows g and g+8
    uint2 q0[4], q1[4];  // quant bytes [32c + 8t, +8) of each chunk c, rows g and g+8
};
template <int WT>
struct MmaW : MmaWBase {};
template <>
struct MmaW<GGUF_Q5_K> : MmaWBase {
    uint2 qh0, qh1;      // high-bit bytes [8t, +8) of rows g and g+8
};

// WT: Q4_K or Q5_K; NT: n-tiles of 8 tokens (8*NT tokens at most)
template <int WT, int NT>
__global__ void __launch_bounds__(NT == 1 ? 512 : 256, 1)
    mmvq_mma_kq_kernel(const MmvqSegs sg, int64_t k, int64_t rb, const uint8_t *__restrict__ xq, int m_act, int yt,
                       int grp) {
    constexpr int TOK = 8 * NT;
    constexpr bool Q5 = WT == GGUF_Q5_K;
    constexpr int SB_BYTES = Q5 ? Q5_K_BYTES : Q4_K_BYTES;
    constexpr int QOFF = Q5 ? 48 : 16;   // the quant bytes follow the header (and Q5_K's 32 high-bit bytes)
    const int64_t n = sg.rows();
    extern __shared__ __align__(16) uint8_t smem[];
    const int nw = blockDim.x >> 5;
    const MmaSmem L = mma_smem_layout(k, nw, grp, NT);
    uint8_t *xs = smem + L.xs;
    float *da = reinterpret_cast<float *>(smem + L.da);
    uint32_t *saf = reinterpret_cast<uint32_t *>(smem + L.saf);
    float4 *red = reinterpret_cast<float4 *>(smem + L.red);

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    const int nblk = (int)(k / 32), nsb = (int)(k / 256);
    const int64_t xrb = (int64_t)nblk * Q8_1_BYTES;
    const int pitch = (int)L.xs_pitch;
    const int64_t n_tiles = (n + 15) / 16;
    const int sb_lo = warp * nsb / nw, sb_hi = (warp + 1) * nsb / nw;

    // per-thread Q4_K scale selectors for sub-blocks 2t, 2t+1 (see Q4KPiece::pos)
    const Q4KPiece::Pos sel = Q4KPiece::pos(t);

    // row base pointers of the tile being loaded (looked up once per tile)
    int64_t cached_tile = -1;
    const uint8_t *base0 = nullptr, *base1 = nullptr;
    auto load_item = [&](MmaW<WT> &W, int64_t tile, int sb) {
        if (tile != cached_tile) {
            const int64_t r0 = tile * 16 + g, r1 = r0 + 8;
            base0 = seg_row(sg, r0 < n ? r0 : n - 1, rb);
            base1 = seg_row(sg, r1 < n ? r1 : n - 1, rb);
            cached_tile = tile;
        }
        const uint8_t *b0 = base0 + sb * SB_BYTES;
        const uint8_t *b1 = base1 + sb * SB_BYTES;
        W.h0 = __ldg(reinterpret_cast<const uint4 *>(b0));
        W.h1 = __ldg(reinterpret_cast<const uint4 *>(b1));
        if constexpr (Q5) {
            W.qh0 = __ldg(reinterpret_cast<const uint2 *>(b0 + 16 + 8 * t));
            W.qh1 = __ldg(reinterpret_cast<const uint2 *>(b1 + 16 + 8 * t));
        }
#pragma unroll
        for (int c = 0; c < 4; c++) {
            W.q0[c] = __ldg(reinterpret_cast<const uint2 *>(b0 + QOFF + 32 * c + 8 * t));
            W.q1[c] = __ldg(reinterpret_cast<const uint2 *>(b1 + QOFF + 32 * c + 8 * t));
        }
    };

    // the first item's weights are requested before waiting for the kernel
    // that wrote the activations
    int64_t tile = blockIdx.x;
    MmaW<WT> wa, wb;
    if (sb_lo < sb_hi && tile < n_tiles) load_item(wa, tile, sb_lo);
    mmvq_pdl_enter(sg.chain);

    // ---- q8_1 rows into shared memory: asynchronous 4-byte copies, all of a
    // thread's in flight at once (quants of block b at b * 40 + 8, the block's
    // (d, s) word into hdr); zeros for the token rows past m_act
    uint32_t *hdr = reinterpret_cast<uint32_t *>(smem + L.hdr);
    for (int i = tid; i < TOK * nblk; i += blockDim.x) {
        const int tok = i / nblk, b = i - tok * nblk;
        uint32_t *dst = reinterpret_cast<uint32_t *>(xs + tok * pitch + b * 40 + 8);
        if (tok < m_act) {
            const uint8_t *src = xq + tok * xrb + (int64_t)b * Q8_1_BYTES;
            cp_async4(hdr + i, src);
#pragma unroll
            for (int j = 0; j < 8; j++) cp_async4(dst + j, src + 4 + 4 * j);
        } else {
            hdr[i] = 0u;
#pragma unroll
            for (int j = 0; j < 8; j++) dst[j] = 0u;
        }
    }
    cp_async_wait_all();
    __syncthreads();
    // d_a as fp32 [block][token] and the s_a pairs of the min-term MMA [sb][nt][lane]
    for (int i = tid; i < nblk * TOK; i += blockDim.x) {
        const int b = i / TOK, tok = i % TOK;
        da[i] = h2f((uint16_t)(hdr[tok * nblk + b] & 0xffffu));
    }
    for (int i = tid; i < nsb * NT * 32; i += blockDim.x) {
        const int s = i / (NT * 32), l = i & 31, tok = 8 * ((i >> 5) % NT) + (l >> 2), tt = l & 3;
        const uint32_t *h = hdr + tok * nblk + s * 8 + 2 * tt;
        saf[i] = (h[0] >> 16) | (h[1] & 0xffff0000u);
    }
    __syncthreads();   // hdr (the reduction area) is free again

    const uint8_t *xg = xs + g * pitch + 8 + 8 * t;   // this lane's B bytes: token 8nt + g, values 8t .. 8t+7
    const __half2 bias = __floats2half2_rn(-1024.0f, -1024.0f);

    // one (tile, super-block) item; partial sums of rows g, g+8 x tokens 8nt + 2t, +1 into acc[nt]
    auto process = [&](const MmaW<WT> &W, int sb, float (&acc)[NT][4]) {
        const float d0 = h2f(W.h0.x & 0xffff), dm0 = h2f(W.h0.x >> 16);
        const float d1 = h2f(W.h1.x & 0xffff), dm1 = h2f(W.h1.x >> 16);
        // (s, m) of sub-blocks 2t, 2t+1 for rows g and g+8 as bytes (s0, s1, m0, m1)
        const uint32_t r0 = __byte_perm(W.h0.y, W.h0.z, sel.sel_r), r1 = __byte_perm(W.h1.y, W.h1.z, sel.sel_r);
        const uint32_t w0 = __byte_perm(W.h0.w, 0u, sel.sel_w), w1 = __byte_perm(W.h1.w, 0u, sel.sel_w);
        const uint32_t sm0 = (r0 & sel.m1) | ((r0 >> 2) & sel.m2) | (w0 & sel.m3) | ((w0 >> 4) & sel.m4);
        const uint32_t sm1 = (r1 & sel.m1) | ((r1 >> 2) & sel.m2) | (w1 & sel.m3) | ((w1 >> 4) & sel.m4);
        // the scales of chunk c are decoded by lane t = c of the quad
        const uint32_t sp = __byte_perm(sm0, sm1, 0x5410);   // s_2t(g), s_2t+1(g), s_2t(g+8), s_2t+1(g+8)
        float u[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
            for (int i = 0; i < 4; i++) u[nt][i] = 0.0f;
#pragma unroll
        for (int c = 0; c < 4; c++) {
            const uint32_t sc = __shfl_sync(0xffffffffu, sp, (lane & ~3) | c);
            const float sl0 = u8f(sc, 0), sh0 = u8f(sc, 1);
            const float sl1 = u8f(sc, 2), sh1 = u8f(sc, 3);
            const int bl = sb * 8 + 2 * c;   // block of the low nibbles; bl + 1 of the high ones
            const uint2 x0 = W.q0[c], x1 = W.q1[c];
            uint32_t lo00 = x0.x & 0x0F0F0F0Fu, lo10 = x1.x & 0x0F0F0F0Fu;
            uint32_t lo01 = x0.y & 0x0F0F0F0Fu, lo11 = x1.y & 0x0F0F0F0Fu;
            uint32_t hi00 = (x0.x >> 4) & 0x0F0F0F0Fu, hi10 = (x1.x >> 4) & 0x0F0F0F0Fu;
            uint32_t hi01 = (x0.y >> 4) & 0x0F0F0F0Fu, hi11 = (x1.y >> 4) & 0x0F0F0F0Fu;
            if constexpr (Q5) {   // fifth bits: bit 2c of each high-bit byte (low nibbles), 2c + 1 (high)
                const uint32_t h00 = W.qh0.x >> (2 * c), h01 = W.qh0.y >> (2 * c);
                const uint32_t h10 = W.qh1.x >> (2 * c), h11 = W.qh1.y >> (2 * c);
                lo00 |= (h00 << 4) & 0x10101010u;
                lo01 |= (h01 << 4) & 0x10101010u;
                lo10 |= (h10 << 4) & 0x10101010u;
                lo11 |= (h11 << 4) & 0x10101010u;
                hi00 |= (h00 << 3) & 0x10101010u;
                hi01 |= (h01 << 3) & 0x10101010u;
                hi10 |= (h10 << 3) & 0x10101010u;
                hi11 |= (h11 << 3) & 0x10101010u;
            }
#pragma unroll
            for (int nt = 0; nt < NT; nt++) {
                const uint2 bL = *reinterpret_cast<const uint2 *>(xg + 8 * nt * pitch + bl * 40);
                const uint2 bH = *reinterpret_cast<const uint2 *>(xg + 8 * nt * pitch + (bl + 1) * 40);
                int sL[4], sH[4];
                mma_16832_s8(sL, lo00, lo10, lo01, lo11, bL.x, bL.y);
                mma_16832_s8(sH, hi00, hi10, hi01, hi11, bH.x, bH.y);
                const float2 dL = *reinterpret_cast<const float2 *>(da + bl * TOK + 8 * nt + 2 * t);
                const float2 dH = *reinterpret_cast<const float2 *>(da + (bl + 1) * TOK + 8 * nt + 2 * t);
                // accumulator i: row g (i < 2) or g+8, token 8nt + 2t + (i & 1)
                u[nt][0] = fmaf(sl0, dL.x * i2f22(sL[0]), u[nt][0]);
                u[nt][1] = fmaf(sl0, dL.y * i2f22(sL[1]), u[nt][1]);
                u[nt][2] = fmaf(sl1, dL.x * i2f22(sL[2]), u[nt][2]);
                u[nt][3] = fmaf(sl1, dL.y * i2f22(sL[3]), u[nt][3]);
                u[nt][0] = fmaf(sh0, dH.x * i2f22(sH[0]), u[nt][0]);
                u[nt][1] = fmaf(sh0, dH.y * i2f22(sH[1]), u[nt][1]);
                u[nt][2] = fmaf(sh1, dH.x * i2f22(sH[2]), u[nt][2]);
                u[nt][3] = fmaf(sh1, dH.y * i2f22(sH[3]), u[nt][3]);
            }
        }
        // min term: A = m_2t, m_2t+1 of rows g, g+8 at k-slots 2t, 2t+1 (exact fp16 integers)
        uint32_t ma0 = __byte_perm(sm0, 0x64u, 0x4342), ma1 = __byte_perm(sm1, 0x64u, 0x4342);
        {
            __half2 h0 = __hadd2(*reinterpret_cast<__half2 *>(&ma0), bias);
            __half2 h1 = __hadd2(*reinterpret_cast<__half2 *>(&ma1), bias);
            ma0 = *reinterpret_cast<uint32_t *>(&h0);
            ma1 = *reinterpret_cast<uint32_t *>(&h1);
        }
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
            float mv[4];
            mma_16816_f16(mv, ma0, ma1, 0u, 0u, saf[(sb * NT + nt) * 32 + lane], 0u);
            acc[nt][0] = fmaf(d0, u[nt][0], acc[nt][0]);
            acc[nt][1] = fmaf(d0, u[nt][1], acc[nt][1]);
            acc[nt][2] = fmaf(d1, u[nt][2], acc[nt][2]);
            acc[nt][3] = fmaf(d1, u[nt][3], acc[nt][3]);
            acc[nt][0] = fmaf(-dm0, mv[0], acc[nt][0]);
            acc[nt][1] = fmaf(-dm0, mv[1], acc[nt][1]);
            acc[nt][2] = fmaf(-dm1, mv[2], acc[nt][2]);
            acc[nt][3] = fmaf(-dm1, mv[3], acc[nt][3]);
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
                for (int j = 0; j < nw; j++) {
                    const float4 v = red[(((buf * grp + tt) * nw + j) * NT + nt) * 32 + l];
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

inline int mma_q4k_warps(int64_t k, int nt) {
    const int cap = nt == 1 ? 16 : 8;   // 512 / 256 threads
    int nw = (int)(k / 256 / 2);
    return nw < 1 ? 1 : nw > cap ? cap : nw;
}
// tiles per reduction group: 4 when shared memory allows, else fewer (0: does not fit)
inline int mma_q4k_group(int64_t k, int nt) {
    for (int grp = 4; grp >= 1; grp /= 2)
        if (mma_smem_layout(k, mma_q4k_warps(k, nt), grp, nt).total <= (int64_t)device_info().smem_optin) return grp;
    return 0;
}
inline int mma_q4k_ntiles(int64_t m) { return m <= 8 ? 1 : m <= 16 ? 2 : 4; }
// whether the tensor-core MMVQ takes m tokens of K-long Q4_K rows (the q8_1
// rows must fit in shared memory; m <= 32)
inline bool mma_q4k_fits(int64_t k, int64_t m) { return m <= 32 && mma_q4k_group(k, mma_q4k_ntiles(m)) > 0; }

template <int WT, int NT>
inline cudaError_t launch_mmvq_mma_kq_nt(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt,
                                         cudaStream_t s) {
    const int64_t n = sg.rows();
    const int nw = mma_q4k_warps(k, NT), grp = mma_q4k_group(k, NT);
    if (grp == 0) return cudaErrorInvalidValue;
    const MmaSmem L = mma_smem_layout(k, nw, grp, NT);
    auto kern = mmvq_mma_kq_kernel<WT, NT>;
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
    const int64_t rb = k / 256 * (int64_t)(WT == GGUF_Q5_K ? Q5_K_BYTES : Q4_K_BYTES);
    return cudaLaunchKernelEx(&cfg, kern, sg, k, rb, xq, (int)m, yt, grp);
}

// Q4_K: 5..32 tokens (1, 2 or 4 n-tiles); Q5_K: 5..8 tokens (one n-tile)
template <int WT>
inline cudaError_t launch_mmvq_mma_kq(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt,
                                      cudaStream_t s) {
    if constexpr (WT == GGUF_Q5_K) {
        return m <= 8 ? launch_mmvq_mma_kq_nt<WT, 1>(sg, k, xq, m, yt, s) : cudaErrorInvalidValue;
    } else {
        switch (mma_q4k_ntiles(m)) {
        case 1: return launch_mmvq_mma_kq_nt<WT, 1>(sg, k, xq, m, yt, s);
        case 2: return launch_mmvq_mma_kq_nt<WT, 2>(sg, k, xq, m, yt, s);
        default: return launch_mmvq_mma_kq_nt<WT, 4>(sg, k, xq, m, yt, s);
        }
    }
}

}  // namespace gg
