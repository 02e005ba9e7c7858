// Tensor-core MMVQ for 5..8 tokens of Q8_0, Q4_0 and MXFP4 weights (32-value
// blocks with one scale each): the per-block int32 dot products of the blockwise
// formula run on warp-level int8 MMAs (mma.sync m16n8k32 s8 x s8 -> s32), one
// MMA per 32-value block of 16 weight rows against 8 tokens, so each s32
// accumulator is exactly the block dot S of one (row, token) pair, and
//   y += d_w * d_a * S
// is applied per block in fp32, as in the dp4a kernel.  Q8_0 quants enter the
// MMA as they are; Q4_0 nibbles enter unsigned (0..15) and MXFP4 codes as the
// biased bytes 16 + k (k = 2 e2m1, -12..12), and the offset comes off the exact
// sum, S = MMA - OFF * sum(q_a) (OFF 8 or 16), with the activation blocks'
// quant sums computed once per CTA.  MXFP4's scale is 2^(e - 128) of the
// block's E8M0 byte e, since its values are k * 2^(e - 128).
//
// The blocks are 34 (Q8_0), 18 (Q4_0) or 17 (MXFP4) bytes, 2-byte aligned or
// not at all, so an item (16 rows x 8 blocks, 16 for MXFP4) is copied into a
// per-warp shared-memory buffer with 16-byte asynchronous copies (an item of a
// 16-byte-aligned row whose K is a multiple of the item starts and ends on
// 16-byte boundaries: 272 / 144 / 272 bytes per row), into a ring of NBUF
// buffers so the next items' copies are in flight while one computes; the
// lanes then read their fragments from there.
// Work split and the q8_1 staging are those of the K-quant tensor-core kernel
// (mmvq_mma.cuh): warp w takes items [w * nsb / NW, (w + 1) * nsb / NW) of
// every 16-row tile, and the warps' partial sums are added in a fixed order.
#pragma once

#include <type_traits>

#include "mmvq_mma.cuh"

namespace gg {

template <int WT>
struct SbTraits;
// BB: block bytes; NB: blocks per item; NBUF: item buffers per warp (NBUF - 1
// items in flight while one computes; Q4_0's smaller buffers let two CTAs
// share an SM); OFF: the offset of the quants entering the MMA
template <>
struct SbTraits<GGUF_Q8_0> {
    static constexpr int BB = Q8_0_BYTES, NB = 8, NBUF = 3, OFF = 0;   // 34-byte blocks
};
template <>
struct SbTraits<GGUF_Q4_0> {
    static constexpr int BB = Q4_0_BYTES, NB = 8, NBUF = 3, OFF = 8;   // 18-byte blocks
};
template <>
struct SbTraits<GGUF_MXFP4> {
    static constexpr int BB = MXFP4_BYTES, NB = 16, NBUF = 3, OFF = 16;   // 17-byte blocks
};

// compile-time loop: f(std::integral_constant<int, I>) for I in [B, N)
template <int B, int N, class F>
__device__ __forceinline__ void unroll_c(F &&f) {
    if constexpr (B < N) {
        f(std::integral_constant<int, B>{});
        unroll_c<B + 1, N>(f);
    }
}

// 4 bytes at a shared-memory address p with p % 4 == O (compile-time):
// aligned words and a funnel shift, reading [p - O, p - O + 8) when O != 0
template <int O>
__device__ __forceinline__ uint32_t lds4_at(const uint8_t *p) {
    if constexpr (O == 0) {
        return *reinterpret_cast<const uint32_t *>(p);
    } else {
        const uint32_t *w = reinterpret_cast<const uint32_t *>(p - O);
        return __funnelshift_r(w[0], w[1], 8 * O);
    }
}

__device__ __forceinline__ void cp_async16(void *sdst, const void *gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(sdst)),
                 "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// wait until at most N of the thread's committed groups are still pending
template <int N>
__device__ __forceinline__ void cp_async_wait_n() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 4 bytes at a shared-memory address that is 4-byte aligned (A4) or 2 mod 4
template <bool A4>
__device__ __forceinline__ uint32_t lds4(const uint8_t *p) {
    if constexpr (A4) {
        return *reinterpret_cast<const uint32_t *>(p);
    } else {
        return (uint32_t)*reinterpret_cast<const uint16_t *>(p) |
               ((uint32_t)*reinterpret_cast<const uint16_t *>(p + 2) << 16);
    }
}

template <int WT>
constexpr int sb_item_bytes_t() { return SbTraits<WT>::NB * SbTraits<WT>::BB; }
inline int sb_nb(int wt) {
    return wt == GGUF_Q8_0 ? SbTraits<GGUF_Q8_0>::NB : wt == GGUF_Q4_0 ? SbTraits<GGUF_Q4_0>::NB : SbTraits<GGUF_MXFP4>::NB;
}
inline int64_t sb_item_bytes(int wt) {
    return wt == GGUF_Q8_0 ? sb_item_bytes_t<GGUF_Q8_0>()
           : wt == GGUF_Q4_0 ? sb_item_bytes_t<GGUF_Q4_0>() : sb_item_bytes_t<GGUF_MXFP4>();
}
inline int sb_nbuf(int wt) {
    return wt == GGUF_Q8_0 ? SbTraits<GGUF_Q8_0>::NBUF
           : wt == GGUF_Q4_0 ? SbTraits<GGUF_Q4_0>::NBUF : SbTraits<GGUF_MXFP4>::NBUF;
}
// warps per CTA: at most 8, and at least one item of every tile each
inline int mma_sb_warps(int wt, int64_t k) {
    const int nsb = (int)(k / (32 * sb_nb(wt)));
    return nsb < 8 ? (nsb < 1 ? 1 : nsb) : 8;
}
// shared memory: the K-quant kernel's activation layout (one n-tile), the
// activation blocks' quant sums times OFF (int32 [block][token]), then the
// per-warp item buffers (NBUF items of 16 rows each)
__host__ __device__ inline int64_t mma_sb_qs_offset(int64_t k, int nw, int grp) {
    return (mma_smem_layout(k, nw, grp, 1).total + 15) / 16 * 16;
}
__host__ __device__ inline int64_t mma_sb_wbuf_offset(int64_t k, int nw, int grp) {
    return mma_sb_qs_offset(k, nw, grp) + (k / 32 * 8 * 4 + 15) / 16 * 16;
}
inline int64_t mma_sb_smem(int wt, int64_t k, int nw, int grp) {
    return mma_sb_wbuf_offset(k, nw, grp) + (int64_t)nw * sb_nbuf(wt) * 16 * sb_item_bytes(wt);
}
// tiles per reduction group: the largest that lets two CTAs share an SM, else
// the largest that fits one (0: does not fit)
inline int mma_sb_group(int wt, int64_t k) {
    const int64_t two = 113 * 1024;   // two CTAs within an SM's 228 KB, 1 KB reserved per CTA
    for (int grp = 4; grp >= 1; grp /= 2)
        if (mma_sb_smem(wt, k, mma_sb_warps(wt, k), grp) <= two) return grp;
    for (int grp = 4; grp >= 1; grp /= 2)
        if (mma_sb_smem(wt, k, mma_sb_warps(wt, k), grp) <= (int64_t)device_info().smem_optin) return grp;
    return 0;
}

template <int WT>
__global__ void __launch_bounds__(256, 2)
    mmvq_mma_sb_kernel(const MmvqSegs sg, int64_t k, int64_t rb, const uint8_t *__restrict__ xq, int m_act, int yt,
                       int grp) {
    constexpr int BB = SbTraits<WT>::BB, NB = SbTraits<WT>::NB, OFF = SbTraits<WT>::OFF;
    constexpr int IB = NB * BB;       // bytes of one row's item
    constexpr int NCH = IB / 16;      // 16-byte chunks of one row's item
    constexpr int TOK = 8;
    constexpr int NBUF = SbTraits<WT>::NBUF;
    const int64_t n = sg.rows();
    extern __shared__ __align__(16) uint8_t smem[];
    const int nw = blockDim.x >> 5;
    const MmaSmem L = mma_smem_layout(k, nw, grp, 1);
    uint8_t *xs = smem + L.xs;
    float *da = reinterpret_cast<float *>(smem + L.da);
    float4 *red = reinterpret_cast<float4 *>(smem + L.red);
    int32_t *qs8 = reinterpret_cast<int32_t *>(smem + mma_sb_qs_offset(k, nw, grp));
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint8_t *wbuf = smem + mma_sb_wbuf_offset(k, nw, grp) + (int64_t)warp * NBUF * 16 * IB;

    const int g = lane >> 2, t = lane & 3;
    const int nblk = (int)(k / 32), nsb = (int)(k / (32 * NB));
    const int64_t xrb = (int64_t)nblk * Q8_1_BYTES;
    const int pitch = (int)L.xs_pitch;
    const int64_t n_tiles = (n + 15) / 16;
    const int sb_lo = warp * nsb / nw, sb_hi = (warp + 1) * nsb / nw;

    // the rows of the tile being copied: lane r < 16 holds row r's base
    // (rows past the matrix read its last row; their results are not stored)
    int64_t ptile = -1;
    uint64_t my_row = 0;
    // copy item (tile, sb) into buffer b: chunk c of the 16 x NCH list is row
    // c / NCH, bytes [16 (c % NCH), +16) of its item
    auto issue = [&](int64_t tile, int sb, int b) {
        if (tile != ptile) {
            const int64_t r = tile * 16 + (lane & 15);
            my_row = reinterpret_cast<uint64_t>(seg_row(sg, r < n ? r : n - 1, rb));
            ptile = tile;
        }
        uint8_t *dst = wbuf + b * 16 * IB;
        // the same trip count in every lane (the shuffle needs all 32)
#pragma unroll
        for (int it = 0; it < (16 * NCH + 31) / 32; it++) {
            const int c = lane + 32 * it;
            const int cc = c < 16 * NCH ? c : 16 * NCH - 1;
            const int row = cc / NCH, j = cc - row * NCH;
            const uint64_t base = __shfl_sync(0xffffffffu, my_row, row);
            if (c < 16 * NCH)
                cp_async16(dst + row * IB + 16 * j, reinterpret_cast<const uint8_t *>(base) + (int64_t)sb * IB + 16 * j);
        }
        cp_async_commit();
    };

    // this warp's items in order: (tile, sb) for sb in [sb_lo, sb_hi), tiles
    // blockIdx.x, + gridDim.x, ...; the copy cursor runs NBUF - 1 items ahead
    // of the compute cursor (an empty group past the end keeps the count)
    int64_t ctile = blockIdx.x;
    int csb = sb_lo, pc = 0;
    auto issue_next = [&]() {
        if (ctile < n_tiles) {
            issue(ctile, csb, pc % NBUF);
            if (++csb >= sb_hi) {
                csb = sb_lo;
                ctile += gridDim.x;
            }
        } else {
            cp_async_commit();
        }
        pc++;
    };
    // the first items' copies go out before waiting for the kernel that wrote
    // the activations
#pragma unroll
    for (int i = 0; i < NBUF - 1; i++) issue_next();
    mmvq_pdl_enter(sg.chain);

    // ---- q8_1 rows into shared memory (as the K-quant kernel, one n-tile)
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
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();
    for (int i = tid; i < nblk * TOK; i += blockDim.x) {
        const int b = i / TOK, tok = i % TOK;
        da[i] = h2f((uint16_t)(hdr[tok * nblk + b] & 0xffffu));
        if constexpr (OFF != 0) {
            const uint32_t *qw = reinterpret_cast<const uint32_t *>(xs + tok * pitch + b * 40 + 8);
            int sum = 0;
#pragma unroll
            for (int j = 0; j < 8; j++) sum = __dp4a((int)qw[j], 0x01010101, sum);
            qs8[i] = OFF * sum;
        }
    }
    __syncthreads();   // hdr (the reduction area) is free again

    const uint8_t *xg = xs + g * pitch + 8;   // token g's quants of block b at xg + 40 b
    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    int gi = 0, rbuf = 0, cc = 0;
    int64_t tile = blockIdx.x;
    int sb = sb_lo;
    while (tile < n_tiles) {
        issue_next();                 // into the buffer computed one item ago
        cp_async_wait_n<NBUF - 1>();  // this item's copies are done
        __syncwarp();

        const uint8_t *w0 = wbuf + (cc % NBUF) * 16 * IB + g * IB;   // row g of the tile
        const uint8_t *w1 = w0 + 8 * IB;                     // row g + 8
        // block B of the item (a compile-time constant, so the alignment of its
        // words in the buffer is known: rows start on 16-byte boundaries)
        auto step = [&](auto bc) {
            constexpr int B = decltype(bc)::value;
            const int blk = sb * NB + B;
            float dw0, dw1;
            uint32_t a0, a1, a2, a3, b0, b1;
            if constexpr (WT == GGUF_MXFP4) {
                dw0 = e8m0_half(w0[B * BB]);
                dw1 = e8m0_half(w1[B * BB]);
                // code bytes 4t .. 4t+3 (values 4t.. low, 16+4t.. high) as biased bytes in
                // the order (4t, 16+4t, 4t+1, 17+4t), (4t+2, 18+4t, 4t+3, 19+4t)
                constexpr int O = (B * BB + 1) & 3;
                const uint32_t c0 = lds4_at<O>(w0 + B * BB + 1 + 4 * t);
                const uint32_t c1 = lds4_at<O>(w1 + B * BB + 1 + 4 * t);
                a0 = mxfp4_biased4(c0);
                a2 = mxfp4_biased4(c0 >> 16);
                a1 = mxfp4_biased4(c1);
                a3 = mxfp4_biased4(c1 >> 16);
                const uint32_t x0 = *reinterpret_cast<const uint32_t *>(xg + blk * 40 + 4 * t);
                const uint32_t x1 = *reinterpret_cast<const uint32_t *>(xg + blk * 40 + 16 + 4 * t);
                b0 = __byte_perm(x0, x1, 0x5140);
                b1 = __byte_perm(x0, x1, 0x7362);
            } else {
                dw0 = h2f(*reinterpret_cast<const uint16_t *>(w0 + B * BB));
                dw1 = h2f(*reinterpret_cast<const uint16_t *>(w1 + B * BB));
                // the quant words are 4-byte aligned for odd B (34 B + 2 and 18 B + 2)
                constexpr bool A4 = ((B * BB + 2) & 3) == 0;
                if constexpr (WT == GGUF_Q8_0) {
                    // quants 8t .. 8t+7 of the block (the same K order on both sides)
                    a0 = lds4<A4>(w0 + B * BB + 2 + 8 * t);
                    a2 = lds4<A4>(w0 + B * BB + 6 + 8 * t);
                    a1 = lds4<A4>(w1 + B * BB + 2 + 8 * t);
                    a3 = lds4<A4>(w1 + B * BB + 6 + 8 * t);
                    const uint2 bx = *reinterpret_cast<const uint2 *>(xg + blk * 40 + 8 * t);
                    b0 = bx.x;
                    b1 = bx.y;
                } else {
                    // nibble bytes 4t .. 4t+3: values 4t.. (low) and 16+4t.. (high), unsigned
                    const uint32_t q0 = lds4<A4>(w0 + B * BB + 2 + 4 * t);
                    const uint32_t q1 = lds4<A4>(w1 + B * BB + 2 + 4 * t);
                    a0 = q0 & 0x0F0F0F0Fu;
                    a1 = q1 & 0x0F0F0F0Fu;
                    a2 = (q0 >> 4) & 0x0F0F0F0Fu;
                    a3 = (q1 >> 4) & 0x0F0F0F0Fu;
                    b0 = *reinterpret_cast<const uint32_t *>(xg + blk * 40 + 4 * t);
                    b1 = *reinterpret_cast<const uint32_t *>(xg + blk * 40 + 16 + 4 * t);
                }
            }
            int S[4];
            mma_16832_s8(S, a0, a1, a2, a3, b0, b1);
            if constexpr (OFF != 0) {   // the offset of every weight quant
                const int2 qo = *reinterpret_cast<const int2 *>(qs8 + blk * TOK + 2 * t);
                S[0] -= qo.x;
                S[1] -= qo.y;
                S[2] -= qo.x;
                S[3] -= qo.y;
            }
            const float2 dd = *reinterpret_cast<const float2 *>(da + blk * TOK + 2 * t);
            // accumulator i: row g (i < 2) or g+8, token 2t + (i & 1)
            acc[0] = fmaf(dw0 * dd.x, i2f22(S[0]), acc[0]);
            acc[1] = fmaf(dw0 * dd.y, i2f22(S[1]), acc[1]);
            acc[2] = fmaf(dw1 * dd.x, i2f22(S[2]), acc[2]);
            acc[3] = fmaf(dw1 * dd.y, i2f22(S[3]), acc[3]);
        };
        unroll_c<0, NB>(step);
        __syncwarp();   // every lane is done with this buffer before it is refilled
        cc++;

        if (sb + 1 < sb_hi) {
            sb++;
            continue;
        }
        // the last of this warp's items of the tile: its partial sums
        red[((rbuf * grp + gi) * nw + warp) * 32 + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
        gi++;
        // every `grp` tiles (and after the last), sum the warps' partial
        // results of the group's tiles in a fixed order
        if (gi == grp || tile + gridDim.x >= n_tiles) {
            __syncthreads();
            for (int i = tid; i < gi * 128; i += blockDim.x) {   // per tile: 16 rows x 8 tokens
                const int tt = i >> 7, l = (i >> 2) & 31, e = i & 3;
                float s = 0.0f;
                for (int j = 0; j < nw; j++) {
                    const float4 v = red[((rbuf * grp + tt) * nw + j) * 32 + l];
                    s += e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
                }
                const int64_t t_of = tile - (int64_t)(gi - 1 - tt) * gridDim.x;
                const int64_t row = t_of * 16 + (l >> 2) + 8 * (e >> 1);
                const int tok = 2 * (l & 3) + (e & 1);
                if (row < n && tok < m_act) seg_store(sg, yt, tok, row, s);
            }
            rbuf ^= 1;
            gi = 0;
        }
        tile += gridDim.x;
        sb = sb_lo;
    }
    cp_async_wait_all();   // no copy outlives the CTA
}

// whether 5..8 tokens of K-long rows of type wt (Q8_0 / Q4_0 / MXFP4) can take
// this kernel: whole items, every segment's rows 16-byte aligned, the buffers
// in shared memory
inline bool mma_sb_fits(int wt, const MmvqSegs &sg, int64_t k, int64_t m) {
    if (m > 8 || k % (32 * sb_nb(wt)) != 0) return false;
    for (int i = 0; i < sg.nseg; i++)
        if (reinterpret_cast<uintptr_t>(sg.w[i]) % 16 != 0) return false;
    return mma_sb_group(wt, k) > 0;
}

template <int WT>
inline cudaError_t launch_mmvq_mma_sb(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt,
                                      cudaStream_t s) {
    const int64_t n = sg.rows();
    const int nw = mma_sb_warps(WT, k), grp = mma_sb_group(WT, k);
    if (grp == 0) return cudaErrorInvalidValue;
    const size_t smem = (size_t)mma_sb_smem(WT, k, nw, grp);
    auto kern = mmvq_mma_sb_kernel<WT>;
    cudaError_t e = cudaSuccess;
    const int per_sm = kernel_occupancy(reinterpret_cast<const void *>(kern), nw * 32, smem, &e);
    if (per_sm == 0) return e;
    const int64_t n_tiles = (n + 15) / 16;
    int64_t grid = (int64_t)device_info().sm_count * per_sm;
    if (grid > n_tiles) grid = n_tiles;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)(nw * 32));
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, sg, k, k / 32 * (int64_t)SbTraits<WT>::BB, xq, (int)m, yt, grp);
}

}  // namespace gg
