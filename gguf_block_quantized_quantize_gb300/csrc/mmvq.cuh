// MMVQ: quantized weight x q8_1 activation product for small token counts
// (decode).  y[m][n] = sum over the row's sub-blocks of an exact int32 block
// dot product combined with the fp32 block scales:
//   Q8_0, Q4_0: d_w * d_a * S          (Q4_0: S over q - 8)
//   MXFP4:      2^(e - 128) * d_a * S  (S over k = 2 * e2m1(q))
//   Q4_K, Q5_K: d * s_j * d_a * S_j - dmin * m_j * s_a
//   Q6_K:       d * sc_j * d_a * S_j
// (FreeToken PR #690 "serve GGUF checkpoints on vendored ggml-cuda kernels",
// section "Vendored ggml": q8_1 activations, fp32 accumulation, results in the
// activation dtype; MMVQ serves the small batches, section "Changes").
//
// GB300 design.  The kernel is bound by the HBM read of the packed weights
// (transformers PR #45977 "GgufLinear ...", section "What made it fast": a
// bandwidth-bound decode), so every weight byte is read exactly once, with
// coalesced loads, and the arithmetic per byte is kept small enough to hide
// under those loads:
//   * K is split across the threads of a CTA: thread t owns "piece" t of every
//     row (64 values for the K-quants, Q4_0 and MXFP4, 32 for Q8_0).  Its q8_1 activation quants
//     for that piece are loaded once into registers and reused for every row
//     the CTA visits, so activations cost no bandwidth in the row loop.  For
//     8 tokens, two threads share a piece and take 4 tokens each, which halves
//     the activation registers.
//   * A persistent grid (as many CTAs as fit on the SMs) walks the rows R at a
//     time.  The weights of the next R rows are loaded into registers before
//     the current R rows are computed (two register sets used in turn), so a
//     load is always in flight; the first rows are requested before the kernel
//     waits for the kernel that produced the activations (programmatic
//     dependent launch).
//   * Per-piece int32 sums use dp4a; partial sums of the R x M outputs are
//     reduced with a butterfly (one shuffle per value and level) and across
//     warps through shared memory in a fixed order, so results are
//     deterministic.
#pragma once

#include "common.cuh"
#include "internal.h"
#include "tc.cuh"

namespace gg {

// ---------------------------------------------------------------- Q8_0 pieces
// A Q8_0 piece is one 32-value block; its activations are the matching q8_1
// block: 8 quant words and d_a.
template <int M>
struct ActPiece {
    int q[M][8];      // activation quants of the piece, 4 per word, in piece order
    float f[M];       // d_a
};

template <int M>
__device__ __forceinline__ void load_act_q8_0(ActPiece<M> &a, const uint8_t *xq, int64_t xrb, int m_act, int64_t p,
                                              bool valid) {
#pragma unroll
    for (int mm = 0; mm < M; mm++) {
#pragma unroll
        for (int i = 0; i < 8; i++) a.q[mm][i] = 0;
        a.f[mm] = 0.0f;
        if (!valid || mm >= m_act) continue;
        const uint8_t *blk = xq + mm * xrb + p * Q8_1_BYTES;
        a.f[mm] = h2f(ld_u16(blk));
#pragma unroll
        for (int i = 0; i < 8; i++) a.q[mm][i] = (int)ld_u32(blk + 4 + 4 * i);
    }
}

// Programmatic dependent launch of an MMVQ kernel.  chain 0 (alone): let the
// next kernel launch, then wait for the kernel that wrote the activations.
// chain 1 (first of a batch): wait first, then let the batch's next kernel
// launch: its inputs were written before the batch, so it may read them at
// once.  chain 2 (later in a batch): let the next launch and read at once.
// The batch ends with an ordinary launch of an empty kernel, which starts only
// after every kernel before it has completed.
__device__ __forceinline__ void mmvq_pdl_enter(int chain) {
    if (chain == 1) {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    } else if (chain == 2) {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    } else {
        asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
        asm volatile("griddepcontrol.wait;" ::: "memory");
    }
}

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



// Butterfly over the lanes that share lane % TG (offsets 16 .. TG): V values in,
// one total out; `idx` receives the value index whose total this lane holds.
template <int V, int TG>
__device__ __forceinline__ float butterfly_tg(float (&v)[V], int lane, int &idx) {
    idx = 0;
    int c = V;
#pragma unroll
    for (int o = 16; o >= TG; o >>= 1) {
        if (c > 1) {
            const bool upper = (lane & o) != 0;
#pragma unroll
            for (int j = 0; j < V / 2; j++) {
                if (j < c / 2) {
                    const float send = upper ? v[j] : v[j + c / 2];
                    const float keep = upper ? v[j + c / 2] : v[j];
                    v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
                }
            }
            if (upper) idx += c / 2;
            c /= 2;
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
        }
    }
    return v[0];
}

// lanes that write the totals after butterfly_tg: the lane bits used by the
// plain (non-splitting) levels are zero
template <int V, int TG>
__device__ __forceinline__ bool butterfly_writer(int lane) {
    int c = V, mask = 0;
#pragma unroll
    for (int o = 16; o >= TG; o >>= 1) {
        if (c > 1) c /= 2;
        else mask |= o;
    }
    return (lane & mask) == 0;
}

// ---------------------------------------------------------------- weight segments

// segment of launch row r (end[] is padded with INT64_MAX, so no bound check)
__device__ __forceinline__ int seg_index(const MmvqSegs &sg, int64_t r) {
    int s = 0;
#pragma unroll
    for (int i = 0; i < MMVQ_MAX_SEGS - 1; i++) s += r >= sg.end[i] ? 1 : 0;
    return s;
}
__device__ __forceinline__ const uint8_t *seg_row(const MmvqSegs &sg, int64_t r, int64_t rb) {
    const int s = seg_index(sg, r);
    return sg.w[s] + (r - (s ? sg.end[s - 1] : 0)) * rb;
}
__device__ __forceinline__ void seg_store(const MmvqSegs &sg, int yt, int tok, int64_t r, float v) {
    const int s = seg_index(sg, r);
    store_out(sg.y[s], yt, (int64_t)tok * sg.ldy[s] + (r - (s ? sg.end[s - 1] : 0)), v);
}

// ---------------------------------------------------------------- piece traits
// Each traits type describes one thread's piece of a weight row: where its
// bytes are (Pos, computed once), the raw bytes of one row (W, loaded before
// any arithmetic so several rows are in flight), the activation values of the
// piece for M tokens (A, loaded once), and the block-dot arithmetic.

// 16 bytes at a 2-byte-aligned shared-memory address as four words (aligned
// words plus a funnel shift when p % 4 == 2)
__device__ __forceinline__ void lds16_a2(const uint8_t *p, uint32_t (&o)[4]) {
    const uint32_t *b = reinterpret_cast<const uint32_t *>(reinterpret_cast<uintptr_t>(p) & ~uintptr_t(3));
    const int sh = (reinterpret_cast<uintptr_t>(p) & 2) ? 16 : 0;
    uint32_t w[5];
#pragma unroll
    for (int i = 0; i < 5; i++) w[i] = b[i];
#pragma unroll
    for (int i = 0; i < 4; i++) o[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

// Q8_0 with staged loads: a warp's 32 pieces are 32 consecutive blocks, one
// contiguous span of up to 1088 bytes.  As for Q6_K (below), the span is read
// with 16-byte loads of its 16-byte-aligned cover plus 2-byte loads of a tail,
// written to the warp's shared-memory buffer, and each lane takes its block's
// d and quants from there.
struct Q80Piece {
    static constexpr int VALUES = 32;
    static constexpr bool STAGED = true;
    static constexpr int STAGE_CHUNKS = 70;   // 16-byte chunks of a warp's buffer (1088 + 15 bytes)
    struct Pos {
        int64_t p;       // piece = block index in the row
        int lane;
        int span_off;    // byte offset of the warp's span in the row
        int span_len;    // bytes of the span (32 / TG blocks, fewer at the end of the row)
        int fld;         // byte offset of the piece's block in the span
    };
    struct W { uint4 c[3]; uint32_t t; uint32_t head; };
    struct Wf { uint32_t q[8]; uint32_t d; };
    template <int M> using A = ActPiece<M>;
    // piece p, thread tg of its TG: the warp holds pieces [PW w, PW w + PW), PW = 32 / TG
    template <int TG>
    static __device__ __forceinline__ Pos pos(int64_t p, int tg, int64_t k) {
        constexpr int PW = 32 / TG;
        const int64_t w = p / PW, left = k / 32 - PW * w;
        Pos q;
        q.p = p;
        q.lane = (int)((p * TG + tg) & 31);
        q.span_off = (int)(w * PW * Q8_0_BYTES);
        q.span_len = (int)((left < PW ? (left > 0 ? left : 0) : PW) * Q8_0_BYTES);
        q.fld = (int)(p % PW) * Q8_0_BYTES;
        return q;
    }
    static __device__ __forceinline__ void load(W &w, const uint8_t *row, const Pos &q) {
        const uint8_t *a = row + q.span_off;
        const uint32_t head = (uint32_t)(reinterpret_cast<uintptr_t>(a) & 15);
        const uint4 *c0 = reinterpret_cast<const uint4 *>(a - head);
        const int full = (int)(head + q.span_len) >> 4;
#pragma unroll
        for (int i = 0; i < 3; i++) {
            const int c = q.lane + 32 * i;
            w.c[i] = c < full ? __ldg(c0 + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        const int tail = (int)((head + q.span_len) & 15) >> 1;
        w.t = q.lane < tail ? ld_u16(reinterpret_cast<const uint8_t *>(c0 + full) + 2 * q.lane) : 0u;
        w.head = head;
    }
    static __device__ __forceinline__ void prepare(const W &w, const Pos &q, uint4 *buf, Wf &f) {
        const int full = (int)(w.head + q.span_len) >> 4;
#pragma unroll
        for (int i = 0; i < 3; i++) {
            const int c = q.lane + 32 * i;
            if (c < full) buf[c] = w.c[i];
        }
        const int tail = (int)((w.head + q.span_len) & 15) >> 1;
        if (q.lane < tail) reinterpret_cast<uint16_t *>(buf + full)[q.lane] = (uint16_t)w.t;
        __syncwarp();
        const uint8_t *blk = reinterpret_cast<const uint8_t *>(buf) + w.head + q.fld;
        f.d = *reinterpret_cast<const uint16_t *>(blk);
        uint32_t lo[4], hi[4];
        lds16_a2(blk + 2, lo);
        lds16_a2(blk + 18, hi);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            f.q[i] = lo[i];
            f.q[4 + i] = hi[i];
        }
        __syncwarp();   // every lane holds its block before the buffer is rewritten
    }
    template <int M>
    static __device__ __forceinline__ void load_act(A<M> &a, const uint8_t *xq, int64_t xrb, int m_act,
                                                    const Pos &q, bool valid) {
        load_act_q8_0<M>(a, xq, xrb, m_act, valid ? q.p : 0, valid);
    }
    template <int M>
    static __device__ __forceinline__ void dot(const Wf &w, const A<M> &a, const Pos &, float (&acc)[M]) {
        const float d = h2f((uint16_t)w.d);
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
            int S = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) S = dp4a_ss((int)w.q[i], a.q[mm][i], S);
            acc[mm] = fmaf(d * a.f[mm], i2f22(S), acc[mm]);
        }
    }
};

// Q4_0 with staged loads, as Q8_0, two blocks per piece: piece p is blocks 2p
// and 2p + 1 (the second absent at the end of a row of an odd number of
// blocks), so a warp's 32 pieces are 64 consecutive 18-byte blocks (only
// 2-byte aligned), one contiguous span of up to 1152 bytes read with 16-byte
// loads of its aligned cover plus 2-byte loads of a tail.  The offset 8 of
// the quants enters the exact integer sum through the activation block's
// quant sum: S = sum(q * q_a) - 8 * sum(q_a).
struct Q40Piece {
    static constexpr int VALUES = 64;
    static constexpr bool STAGED = true;
    static constexpr int STAGE_CHUNKS = 74;   // 16-byte chunks of a warp's buffer (1152 + 14 bytes, + reads)
    struct Pos {
        int64_t p;       // piece: blocks 2p, 2p + 1 of the row
        int lane;
        int span_off;    // byte offset of the warp's span in the row
        int span_len;    // bytes of the span (64 / TG blocks, fewer at the end of the row)
        int fld;         // byte offset of the piece's first block in the span
        bool two;        // block 2p + 1 exists
    };
    struct W { uint4 c[3]; uint32_t t; uint32_t head; };
    struct Wf { uint32_t q[8]; uint32_t d; };   // quants of both blocks; d = d0 | d1 << 16
    template <int M>
    struct A {
        int q[M][16];    // activation quants of both blocks, 4 per word
        float f[M][2];   // d_a of each block
        int sum[M][2];   // 8 * sum of each block's quants
    };
    template <int TG>
    static __device__ __forceinline__ Pos pos(int64_t p, int tg, int64_t k) {
        constexpr int PW = 32 / TG, BW = 2 * PW;   // pieces, blocks per warp
        const int64_t nb = k / 32, w = p / PW, left = nb - BW * w;   // blocks of the row from the span start
        Pos q;
        q.p = p;
        q.lane = (int)((p * TG + tg) & 31);
        q.span_off = (int)(w * BW * Q4_0_BYTES);
        q.span_len = (int)((left < BW ? (left > 0 ? left : 0) : BW) * Q4_0_BYTES);
        q.fld = (int)(p % PW) * 2 * Q4_0_BYTES;
        q.two = 2 * p + 1 < nb;
        return q;
    }
    static __device__ __forceinline__ void load(W &w, const uint8_t *row, const Pos &q) {
        const uint8_t *a = row + q.span_off;
        const uint32_t head = (uint32_t)(reinterpret_cast<uintptr_t>(a) & 15);
        const uint4 *c0 = reinterpret_cast<const uint4 *>(a - head);
        const int full = (int)(head + q.span_len) >> 4;
#pragma unroll
        for (int i = 0; i < 3; i++) {
            const int c = q.lane + 32 * i;
            w.c[i] = c < full ? __ldg(c0 + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        const int tail = (int)((head + q.span_len) & 15) >> 1;
        w.t = q.lane < tail ? ld_u16(reinterpret_cast<const uint8_t *>(c0 + full) + 2 * q.lane) : 0u;
        w.head = head;
    }
    static __device__ __forceinline__ void prepare(const W &w, const Pos &q, uint4 *buf, Wf &f) {
        const int full = (int)(w.head + q.span_len) >> 4;
#pragma unroll
        for (int i = 0; i < 3; i++) {
            const int c = q.lane + 32 * i;
            if (c < full) buf[c] = w.c[i];
        }
        const int tail = (int)((w.head + q.span_len) & 15) >> 1;
        if (q.lane < tail) reinterpret_cast<uint16_t *>(buf + full)[q.lane] = (uint16_t)w.t;
        __syncwarp();
        const uint8_t *blk = reinterpret_cast<const uint8_t *>(buf) + w.head + q.fld;
        uint32_t lo[4], hi[4];
        lds16_a2(blk + 2, lo);
        lds16_a2(blk + 20, hi);
        const uint32_t d0 = *reinterpret_cast<const uint16_t *>(blk);
        const uint32_t d1 = *reinterpret_cast<const uint16_t *>(blk + 18);
        // an absent second block (bytes past the span) contributes nothing
        f.d = d0 | ((q.two ? d1 : 0u) << 16);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            f.q[i] = lo[i];
            f.q[4 + i] = q.two ? hi[i] : 0u;
        }
        __syncwarp();   // every lane holds its blocks before the buffer is rewritten
    }
    template <int M>
    static __device__ __forceinline__ void load_act(A<M> &a, const uint8_t *xq, int64_t xrb, int m_act,
                                                    const Pos &q, bool valid) {
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
#pragma unroll
            for (int b = 0; b < 2; b++) {
                const bool on = valid && mm < m_act && (b == 0 || q.two);
                const uint8_t *blk = xq + mm * xrb + (on ? 2 * q.p + b : 0) * Q8_1_BYTES;
                a.f[mm][b] = on ? h2f(ld_u16(blk)) : 0.0f;
                int sum = 0;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    const int v = on ? (int)ld_u32(blk + 4 + 4 * i) : 0;
                    a.q[mm][8 * b + i] = v;
                    sum = dp4a_ss(v, 0x01010101, sum);
                }
                a.sum[mm][b] = 8 * sum;
            }
        }
    }
    template <int M>
    static __device__ __forceinline__ void dot(const Wf &w, const A<M> &a, const Pos &, float (&acc)[M]) {
        const float d[2] = {h2f((uint16_t)(w.d & 0xffff)), h2f((uint16_t)(w.d >> 16))};
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            lo[i] = w.q[i] & 0x0F0F0F0Fu;          // values 4i .. 4i+3 of the block
            hi[i] = (w.q[i] >> 4) & 0x0F0F0F0Fu;   // values 16 + 4i ..
        }
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
            float v = acc[mm];
#pragma unroll
            for (int b = 0; b < 2; b++) {
                int S = -a.sum[mm][b];
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    S = dp4a_us(lo[4 * b + i], a.q[mm][8 * b + i], S);
                    S = dp4a_us(hi[4 * b + i], a.q[mm][8 * b + 4 + i], S);
                }
                v = fmaf(d[b] * a.f[mm][b], i2f22(S), v);
            }
            acc[mm] = v;
        }
    }
};

// 16 bytes at any shared-memory address as four words (aligned words plus a
// funnel shift)
__device__ __forceinline__ void lds16_a1(const uint8_t *p, uint32_t (&o)[4]) {
    const uint32_t *b = reinterpret_cast<const uint32_t *>(reinterpret_cast<uintptr_t>(p) & ~uintptr_t(3));
    const int sh = 8 * (int)(reinterpret_cast<uintptr_t>(p) & 3);
    uint32_t w[5];
#pragma unroll
    for (int i = 0; i < 5; i++) w[i] = b[i];
#pragma unroll
    for (int i = 0; i < 4; i++) o[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

// MXFP4 as Q4_0: two 17-byte blocks per piece (the second absent at the end of
// a row of an odd number of blocks), a warp's 64 blocks staged as one span of
// up to 1088 bytes; the blocks have no alignment at all, so the span's tail
// is read byte by byte.  Codes become biased bytes 16 + k (mxfp4_biased4), in
// the order (l, l + 16, l + 1, l + 17) that one 16-bit selector gives; the
// activation words are interleaved the same way once, when they are loaded,
// and S = sum((16 + k) * q_a) - 16 * sum(q_a) is exact.
struct MX4Piece {
    static constexpr int VALUES = 64;
    static constexpr bool STAGED = true;
    static constexpr int STAGE_CHUNKS = 72;   // 16-byte chunks of a warp's buffer (1088 + 15 bytes, + reads)
    using Pos = Q40Piece::Pos;
    struct W { uint4 c[3]; uint32_t t; uint32_t head; };
    struct Wf { uint32_t q[8]; uint32_t e; };   // code words of both blocks; e = e0 | e1 << 8
    template <int M>
    struct A {
        int q[M][16];    // activation quants of both blocks, interleaved as the biased codes
        float f[M][2];   // d_a of each block
        int sum[M][2];   // 16 * sum of each block's quants
    };
    template <int TG>
    static __device__ __forceinline__ Pos pos(int64_t p, int tg, int64_t k) {
        constexpr int PW = 32 / TG, BW = 2 * PW;
        const int64_t nb = k / 32, w = p / PW, left = nb - BW * w;
        Pos q;
        q.p = p;
        q.lane = (int)((p * TG + tg) & 31);
        q.span_off = (int)(w * BW * MXFP4_BYTES);
        q.span_len = (int)((left < BW ? (left > 0 ? left : 0) : BW) * MXFP4_BYTES);
        q.fld = (int)(p % PW) * 2 * MXFP4_BYTES;
        q.two = 2 * p + 1 < nb;
        return q;
    }
    static __device__ __forceinline__ void load(W &w, const uint8_t *row, const Pos &q) {
        const uint8_t *a = row + q.span_off;
        const uint32_t head = (uint32_t)(reinterpret_cast<uintptr_t>(a) & 15);
        const uint4 *c0 = reinterpret_cast<const uint4 *>(a - head);
        const int full = (int)(head + q.span_len) >> 4;
#pragma unroll
        for (int i = 0; i < 3; i++) {
            const int c = q.lane + 32 * i;
            w.c[i] = c < full ? __ldg(c0 + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        const int tail = (int)((head + q.span_len) & 15);   // bytes
        w.t = q.lane < tail ? (uint32_t)reinterpret_cast<const uint8_t *>(c0 + full)[q.lane] : 0u;
        w.head = head;
    }
    static __device__ __forceinline__ void prepare(const W &w, const Pos &q, uint4 *buf, Wf &f) {
        const int full = (int)(w.head + q.span_len) >> 4;
#pragma unroll
        for (int i = 0; i < 3; i++) {
            const int c = q.lane + 32 * i;
            if (c < full) buf[c] = w.c[i];
        }
        const int tail = (int)((w.head + q.span_len) & 15);
        if (q.lane < tail) reinterpret_cast<uint8_t *>(buf + full)[q.lane] = (uint8_t)w.t;
        __syncwarp();
        const uint8_t *blk = reinterpret_cast<const uint8_t *>(buf) + w.head + q.fld;
        uint32_t lo[4], hi[4];
        lds16_a1(blk + 1, lo);
        lds16_a1(blk + 1 + MXFP4_BYTES, hi);
        f.e = (uint32_t)blk[0] | ((uint32_t)blk[MXFP4_BYTES] << 8);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            f.q[i] = lo[i];
            f.q[4 + i] = hi[i];   // an absent second block meets zero activations
        }
        __syncwarp();   // every lane holds its blocks before the buffer is rewritten
    }
    template <int M>
    static __device__ __forceinline__ void load_act(A<M> &a, const uint8_t *xq, int64_t xrb, int m_act,
                                                    const Pos &q, bool valid) {
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
#pragma unroll
            for (int b = 0; b < 2; b++) {
                const bool on = valid && mm < m_act && (b == 0 || q.two);
                const uint8_t *blk = xq + mm * xrb + (on ? 2 * q.p + b : 0) * Q8_1_BYTES;
                a.f[mm][b] = on ? h2f(ld_u16(blk)) : 0.0f;
                int x[8], sum = 0;
#pragma unroll
                for (int i = 0; i < 8; i++) {
                    x[i] = on ? (int)ld_u32(blk + 4 + 4 * i) : 0;
                    sum = dp4a_ss(x[i], 0x01010101, sum);
                }
                // code word j covers values 4j..4j+3 (low nibbles) and 16+4j.. (high):
                // its two selectors give (4j, 16+4j, 4j+1, 17+4j), (4j+2, 18+4j, 4j+3, 19+4j)
#pragma unroll
                for (int j = 0; j < 4; j++) {
                    a.q[mm][8 * b + 2 * j] = (int)__byte_perm((uint32_t)x[j], (uint32_t)x[4 + j], 0x5140);
                    a.q[mm][8 * b + 2 * j + 1] = (int)__byte_perm((uint32_t)x[j], (uint32_t)x[4 + j], 0x7362);
                }
                a.sum[mm][b] = 16 * sum;
            }
        }
    }
    template <int M>
    static __device__ __forceinline__ void dot(const Wf &w, const A<M> &a, const Pos &, float (&acc)[M]) {
        const float d[2] = {e8m0_half(w.e & 0xff), e8m0_half((w.e >> 8) & 0xff)};
        uint32_t u[16];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            u[2 * i] = mxfp4_biased4(w.q[i]);
            u[2 * i + 1] = mxfp4_biased4(w.q[i] >> 16);
        }
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
            float v = acc[mm];
#pragma unroll
            for (int b = 0; b < 2; b++) {
                int S = -a.sum[mm][b];
#pragma unroll
                for (int i = 0; i < 8; i++) S = dp4a_us(u[8 * b + i], a.q[mm][8 * b + i], S);
                v = fmaf(d[b] * a.f[mm][b], i2f22(S), v);
            }
            acc[mm] = v;
        }
    }
};

// Q4_K, 64-value pieces: piece p is chunk c = p%4 of super-block p/4, i.e. the
// 32 quant bytes at 16 + 32c whose low nibbles are sub-block 2c and whose high
// nibbles are sub-block 2c+1 (values 64c .. 64c+63).  One thread loads the
// 16-byte header and the 32 quant bytes with three 16-byte loads.
struct Q4KPiece {
    static constexpr int VALUES = 64;
    static constexpr bool STAGED = false;
    static constexpr int STAGE_CHUNKS = 1;
    struct Pos {
        int64_t off;               // byte offset of the super-block in the row
        int c;                     // chunk
        uint32_t sel_r, sel_w;     // byte_perm selectors for the scale bytes
        uint32_t m1, m2, m3, m4;   // masks that assemble (s0, s1, m0, m1) for this c
    };
    struct W { uint4 h, a, b; };
    template <int M>
    struct A {
        int q[M][16];     // quants of q8_1 blocks 2c and 2c+1 of the super-block
        float f[M][4];    // d_a0, d_a1, s_a0, s_a1
    };
    static __device__ __forceinline__ Pos pos(int64_t p) {
        Pos q;
        q.off = (p >> 2) * Q4_K_BYTES;
        q.c = (int)(p & 3);
        const uint32_t cc = (uint32_t)(q.c & 1);
        // sub-blocks j = 2c, 2c+1 take their 6-bit scale / min from the scale
        // bytes sc[0..11] (header words y = sc[0..3], z = sc[4..7], w = sc[8..11]):
        //   j < 4: s = sc[j] & 63, m = sc[j+4] & 63
        //   j >= 4: s = (sc[j+4] & 15) | (sc[j-4] >> 6) << 4,
        //           m = (sc[j+4] >> 4) | (sc[j] >> 6) << 4
        // r = (y[2cc], y[2cc+1], z[2cc], z[2cc+1]) and wq = (w[2cc], w[2cc+1]) x 2
        // hold every byte either case needs.
        q.sel_r = (2 * cc) | ((2 * cc + 1) << 4) | ((4 + 2 * cc) << 8) | ((5 + 2 * cc) << 12);
        q.sel_w = (2 * cc) | ((2 * cc + 1) << 4) | ((2 * cc) << 8) | ((2 * cc + 1) << 12);
        const bool lo = q.c < 2;
        q.m1 = lo ? 0x3F3F3F3Fu : 0u;
        q.m2 = lo ? 0u : 0x30303030u;
        q.m3 = lo ? 0u : 0x00000F0Fu;
        q.m4 = lo ? 0u : 0x0F0F0000u;
        return q;
    }
    static __device__ __forceinline__ void load(W &w, const uint8_t *row, const Pos &q) {
        const uint8_t *blk = row + q.off;
        w.h = __ldg(reinterpret_cast<const uint4 *>(blk));
        w.a = __ldg(reinterpret_cast<const uint4 *>(blk + 16 + 32 * q.c));
        w.b = __ldg(reinterpret_cast<const uint4 *>(blk + 32 + 32 * q.c));
    }
    template <int M>
    static __device__ __forceinline__ void load_act(A<M> &a, const uint8_t *xq, int64_t xrb, int m_act,
                                                    const Pos &q, bool valid) {
        const int64_t b0 = (q.off / Q4_K_BYTES) * 8 + 2 * q.c;
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
            const bool on = valid && mm < m_act;
            const uint8_t *p0 = xq + mm * xrb + b0 * Q8_1_BYTES, *p1 = p0 + Q8_1_BYTES;
            const uint32_t ds0 = on ? ld_u32(p0) : 0u, ds1 = on ? ld_u32(p1) : 0u;
            a.f[mm][0] = h2f(ds0 & 0xffff);
            a.f[mm][1] = h2f(ds1 & 0xffff);
            a.f[mm][2] = h2f(ds0 >> 16);
            a.f[mm][3] = h2f(ds1 >> 16);
#pragma unroll
            for (int i = 0; i < 8; i++) {
                a.q[mm][i] = on ? (int)ld_u32(p0 + 4 + 4 * i) : 0;
                a.q[mm][8 + i] = on ? (int)ld_u32(p1 + 4 + 4 * i) : 0;
            }
        }
    }
    template <int M>
    static __device__ __forceinline__ void dot(const W &w, const A<M> &a, const Pos &q, float (&acc)[M]) {
        const float d = h2f(w.h.x & 0xffff), dmin = h2f(w.h.x >> 16);
        const uint32_t r = __byte_perm(w.h.y, w.h.z, q.sel_r);
        const uint32_t wq = __byte_perm(w.h.w, 0u, q.sel_w);
        // bytes (s0, s1, m0, m1), each 6 bits
        const uint32_t sm = (r & q.m1) | ((r >> 2) & q.m2) | (wq & q.m3) | ((wq >> 4) & q.m4);
        const float ds0 = d * u8f(sm, 0);
        // high nibbles are used in place (16 * q), so their scale carries 1/16 (exact)
        const float ds1 = d * u8f(sm, 1) * 0.0625f;
        const float fm0 = u8f(sm, 2), fm1 = u8f(sm, 3);
        const uint32_t raw[8] = {w.a.x, w.a.y, w.a.z, w.a.w, w.b.x, w.b.y, w.b.z, w.b.w};
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            lo[i] = raw[i] & 0x0F0F0F0Fu;
            hi[i] = raw[i] & 0xF0F0F0F0u;
        }
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
            int S0 = 0, S1 = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                S0 = dp4a_us(lo[i], a.q[mm][i], S0);
                S1 = dp4a_us(hi[i], a.q[mm][8 + i], S1);
            }
            float v = ds0 * (a.f[mm][0] * i2f22(S0));
            v = fmaf(ds1, a.f[mm][1] * i2f22(S1), v);
            v = fmaf(-dmin, fmaf(fm0, a.f[mm][2], fm1 * a.f[mm][3]), v);
            acc[mm] += v;
        }
    }
};

// Q5_K, 64-value pieces as Q4_K: piece p is chunk c = p%4 of super-block p/4
// (176 bytes, 16-byte aligned): the same 16-byte header, the 32 quant bytes at
// 48 + 32c, and all 32 high-bit bytes at 16, of which the piece takes bits 2c
// (its low-nibble sub-block) and 2c + 1 (its high-nibble one).  Five 16-byte
// loads per piece; the four pieces of a super-block sit in adjacent lanes, so
// a warp still reads each high-bit byte from DRAM once.
struct Q5KPiece {
    static constexpr int VALUES = 64;
    static constexpr bool STAGED = false;
    static constexpr int STAGE_CHUNKS = 1;
    struct Pos {
        int64_t sb;                // super-block index in the row
        int c;                     // chunk
        uint32_t sel_r, sel_w;     // scale-byte selectors, as Q4KPiece
        uint32_t m1, m2, m3, m4;
    };
    struct W { uint4 h, h0, h1, a, b; };
    template <int M> using A = Q4KPiece::A<M>;
    static __device__ __forceinline__ Pos pos(int64_t p) {
        const Q4KPiece::Pos k4 = Q4KPiece::pos(p);
        Pos q;
        q.sb = p >> 2;
        q.c = k4.c;
        q.sel_r = k4.sel_r;
        q.sel_w = k4.sel_w;
        q.m1 = k4.m1;
        q.m2 = k4.m2;
        q.m3 = k4.m3;
        q.m4 = k4.m4;
        return q;
    }
    static __device__ __forceinline__ void load(W &w, const uint8_t *row, const Pos &q) {
        const uint8_t *blk = row + q.sb * Q5_K_BYTES;
        w.h = __ldg(reinterpret_cast<const uint4 *>(blk));
        w.h0 = __ldg(reinterpret_cast<const uint4 *>(blk + 16));
        w.h1 = __ldg(reinterpret_cast<const uint4 *>(blk + 32));
        w.a = __ldg(reinterpret_cast<const uint4 *>(blk + 48 + 32 * q.c));
        w.b = __ldg(reinterpret_cast<const uint4 *>(blk + 64 + 32 * q.c));
    }
    template <int M>
    static __device__ __forceinline__ void load_act(A<M> &a, const uint8_t *xq, int64_t xrb, int m_act,
                                                    const Pos &q, bool valid) {
        Q4KPiece::Pos k4{};
        k4.off = q.sb * Q4_K_BYTES;   // Q4KPiece::load_act locates the q8_1 blocks from off and c
        k4.c = q.c;
        Q4KPiece::load_act<M>(a, xq, xrb, m_act, k4, valid);
    }
    template <int M>
    static __device__ __forceinline__ void dot(const W &w, const A<M> &a, const Pos &q, float (&acc)[M]) {
        const float d = h2f(w.h.x & 0xffff), dmin = h2f(w.h.x >> 16);
        const uint32_t r = __byte_perm(w.h.y, w.h.z, q.sel_r);
        const uint32_t wq = __byte_perm(w.h.w, 0u, q.sel_w);
        const uint32_t sm = (r & q.m1) | ((r >> 2) & q.m2) | (wq & q.m3) | ((wq >> 4) & q.m4);
        const float ds0 = d * u8f(sm, 0);
        const float ds1 = d * u8f(sm, 1);
        const float fm0 = u8f(sm, 2), fm1 = u8f(sm, 3);
        const uint32_t raw[8] = {w.a.x, w.a.y, w.a.z, w.a.w, w.b.x, w.b.y, w.b.z, w.b.w};
        const uint32_t qh[8] = {w.h0.x, w.h0.y, w.h0.z, w.h0.w, w.h1.x, w.h1.y, w.h1.z, w.h1.w};
        const int sh = 2 * q.c;
        uint32_t lo[8], hi[8];
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t hb = qh[i] >> sh;   // bit 0 of each byte: sub-block 2c, bit 1: 2c + 1
            lo[i] = (raw[i] & 0x0F0F0F0Fu) | ((hb << 4) & 0x10101010u);
            hi[i] = ((raw[i] >> 4) & 0x0F0F0F0Fu) | ((hb << 3) & 0x10101010u);
        }
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
            int S0 = 0, S1 = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                S0 = dp4a_us(lo[i], a.q[mm][i], S0);
                S1 = dp4a_us(hi[i], a.q[mm][8 + i], S1);
            }
            float v = ds0 * (a.f[mm][0] * i2f22(S0));
            v = fmaf(ds1, a.f[mm][1] * i2f22(S1), v);
            v = fmaf(-dmin, fmaf(fm0, a.f[mm][2], fm1 * a.f[mm][3]), v);
            acc[mm] += v;
        }
    }
};

// Q6_K blocks (210 bytes) are only 2-byte aligned, so per-thread loads of a
// piece's fields cost many narrow, scattered requests.  Instead the warp's
// span of 8 consecutive blocks of a row (1680 contiguous bytes) is read with
// 16-byte loads of its 16-byte-aligned cover (lane l takes chunks l + 32 i),
// plus 2-byte loads of a tail that does not fill a chunk; `prepare` writes the
// span to the warp's shared-memory buffer and every lane reads its piece's
// fields from there.  Nothing outside the span's row is read except bytes of
// the same aligned chunk before the span start, which belong to the view.
struct Q6KPiece {
    static constexpr int VALUES = 64;
    static constexpr bool STAGED = true;
    static constexpr int STAGE_CHUNKS = 108;   // 16-byte chunks of a warp's buffer (1680 + 15 bytes)
    struct Pos {
        int64_t off;     // byte offset of the piece's block in the row
        int h, l0;       // half of the block, 16-value offset
        int lane;        // lane in the warp
        int span_off;    // byte offset of the warp's span in the row
        int span_len;    // bytes of the span (8 / TG blocks, fewer at the end of the row)
        int fld;         // byte offset of the piece's block in the span
    };
    struct Wf { uint32_t ql0[4], ql1[4], qh[4]; uint32_t sc; uint32_t d; };   // one piece's fields
    struct W { uint4 c[4]; uint32_t t; uint32_t head; };                       // the lane's share of the span
    template <int M>
    struct A {
        int q[M][16];    // run g quants: words 4g .. 4g+3
        float f[M][4];   // d_a of run g
        int sum[M][4];   // 32 * sum of the run's 16 quants
    };
    // piece p, thread tg of its TG: the warp holds pieces [PW w, PW w + PW), PW = 32 / TG,
    // i.e. blocks [PW w / 4, +PW / 4)
    template <int TG>
    static __device__ __forceinline__ Pos pos(int64_t p, int tg, int64_t k) {
        constexpr int PW = 32 / TG, BW = PW / 4;
        const int64_t w = p / PW, left = k / 256 - BW * w;   // blocks of the row from the span start
        Pos q;
        q.off = (p >> 2) * Q6_K_BYTES;
        q.h = (int)((p >> 1) & 1);
        q.l0 = 16 * (int)(p & 1);
        q.lane = (int)((p * TG + tg) & 31);
        q.span_off = (int)(w * BW * Q6_K_BYTES);
        q.span_len = (int)((left < BW ? (left > 0 ? left : 0) : BW) * Q6_K_BYTES);
        q.fld = (int)((p % PW) >> 2) * Q6_K_BYTES;
        return q;
    }
    static __device__ __forceinline__ void load(W &w, const uint8_t *row, const Pos &q) {
        const uint8_t *a = row + q.span_off;
        const uint32_t head = (uint32_t)(reinterpret_cast<uintptr_t>(a) & 15);
        const uint4 *c0 = reinterpret_cast<const uint4 *>(a - head);
        const int full = (int)(head + q.span_len) >> 4;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int c = q.lane + 32 * i;
            w.c[i] = c < full ? __ldg(c0 + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        const int tail = (int)((head + q.span_len) & 15) >> 1;
        w.t = q.lane < tail ? ld_u16(reinterpret_cast<const uint8_t *>(c0 + full) + 2 * q.lane) : 0u;
        w.head = head;
    }
    // the span into the warp's buffer, then this lane's fields out of it
    static __device__ __forceinline__ void prepare(const W &w, const Pos &q, uint4 *buf, Wf &f) {
        const int full = (int)(w.head + q.span_len) >> 4;
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const int c = q.lane + 32 * i;
            if (c < full) buf[c] = w.c[i];
        }
        const int tail = (int)((w.head + q.span_len) & 15) >> 1;
        if (q.lane < tail) reinterpret_cast<uint16_t *>(buf + full)[q.lane] = (uint16_t)w.t;
        __syncwarp();
        const uint8_t *blk = reinterpret_cast<const uint8_t *>(buf) + w.head + q.fld;
        lds16_a2(blk + 64 * q.h + q.l0, f.ql0);
        lds16_a2(blk + 64 * q.h + 32 + q.l0, f.ql1);
        lds16_a2(blk + 128 + 32 * q.h + q.l0, f.qh);
        uint32_t s[3];
        const uint8_t *sp = blk + 192 + 8 * q.h;   // sc[8h .. 8h+7]
        const uint32_t *sb = reinterpret_cast<const uint32_t *>(reinterpret_cast<uintptr_t>(sp) & ~uintptr_t(3));
#pragma unroll
        for (int i = 0; i < 3; i++) s[i] = sb[i];
        const int sh = (reinterpret_cast<uintptr_t>(sp) & 2) ? 16 : 0;
        const uint32_t s0 = __funnelshift_r(s[0], s[1], sh), s1 = __funnelshift_r(s[1], s[2], sh);
        // scales of runs g = 0..3: sc[8h + l0/16 + 2g]
        f.sc = q.l0 ? __byte_perm(s0, s1, 0x7531) : __byte_perm(s0, s1, 0x6420);
        f.d = *reinterpret_cast<const uint16_t *>(blk + 208);
        __syncwarp();   // every lane holds its fields before the buffer is rewritten
    }
    template <int M>
    static __device__ __forceinline__ void load_act(A<M> &a, const uint8_t *xq, int64_t xrb, int m_act,
                                                    const Pos &q, bool valid) {
        const int64_t b0 = (q.off / Q6_K_BYTES) * 8 + 4 * q.h;
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
            const bool on = valid && mm < m_act;
#pragma unroll
            for (int g = 0; g < 4; g++) {
                const uint8_t *blk = xq + mm * xrb + (b0 + g) * Q8_1_BYTES;
                a.f[mm][g] = on ? h2f(ld_u16(blk)) : 0.0f;
                int sum = 0;
#pragma unroll
                for (int i = 0; i < 4; i++) {
                    const int v = on ? (int)ld_u32(blk + 4 + q.l0 + 4 * i) : 0;
                    a.q[mm][4 * g + i] = v;
                    sum = dp4a_ss(v, 0x01010101, sum);
                }
                a.sum[mm][g] = 32 * sum;
            }
        }
    }
    template <int M>
    static __device__ __forceinline__ void dot(const Wf &w, const A<M> &a, const Pos &, float (&acc)[M]) {
        const float d = h2f((uint16_t)w.d);
        float dsc[4];
#pragma unroll
        for (int g = 0; g < 4; g++) dsc[g] = d * i2f22((int)(int8_t)((w.sc >> (8 * g)) & 0xff));
        uint32_t u[4][4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t A0 = w.ql0[i], A1 = w.ql1[i], H = w.qh[i];
            u[0][i] = (A0 & 0x0F0F0F0Fu) | ((H << 4) & 0x30303030u);
            u[1][i] = (A1 & 0x0F0F0F0Fu) | ((H << 2) & 0x30303030u);
            u[2][i] = ((A0 >> 4) & 0x0F0F0F0Fu) | (H & 0x30303030u);
            u[3][i] = ((A1 >> 4) & 0x0F0F0F0Fu) | ((H >> 2) & 0x30303030u);
        }
#pragma unroll
        for (int mm = 0; mm < M; mm++) {
            float v = 0.0f;
#pragma unroll
            for (int g = 0; g < 4; g++) {
                int S = -a.sum[mm][g];
#pragma unroll
                for (int i = 0; i < 4; i++) S = dp4a_us(u[g][i], a.q[mm][4 * g + i], S);
                v = fmaf(dsc[g], a.f[mm][g] * i2f22(S), v);
            }
            acc[mm] += v;
        }
    }
};

// ---------------------------------------------------------------- the kernel
// Thread t of a CTA owns piece t / TG of every row and the tokens
// [(t % TG) * M, +M).  The CTA walks rows [n0, n0 + R) for n0 = blockIdx.x * R,
// + gridDim.x * R, ...
// MULTI: more than one weight segment (row addresses looked up per row group);
// a single segment keeps its pointers in registers.
// ROUTES: MoE route slots, one per grid row (blockIdx.y = r): the weights are
// expert ids[r] of the bank sg.w[0], the activations the q8_1 row of route r
// (or of its token), the fp32 output row r of sg.y[0]; skipped routes
// (pos[r] < 0) exit at once.  M = 1, one segment.  With rt.pack = G > 1 (one
// warp, rows of 32 / G whole pieces) G consecutive rows of the expert, which
// are contiguous, are loaded and staged as one row of G * k values; lane l
// takes piece l % (32 / G) of row l / (32 / G) and the lanes of each row are
// reduced on their own.
template <class PT, int M, int TG, int R, int MAXT, bool MULTI, bool ROUTES = false>
__global__ void __launch_bounds__(MAXT, MAXT == 32 ? 16 : 1) mmvq_kernel(const MmvqSegs sg, int64_t k, int64_t rb,
                                                   const uint8_t *__restrict__ xq, int m_act, int yt,
                                                   const MmvqRoutes rt) {
    const int64_t n = sg.rows();
    const uint8_t *w0 = sg.w[0];
    void *y0 = sg.y[0];
    const int64_t ldy0 = sg.ldy[0];
    if constexpr (ROUTES) {
        static_assert(M == 1 && !MULTI, "routes: one token, one segment");
        // the route table and the activations come from earlier kernels
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int64_t r = blockIdx.y;
        if (rt.pos[r] < 0) return;
        w0 += (int64_t)rt.ids[r] * rt.expert_stride;
        y0 = reinterpret_cast<float *>(y0) + r * n;
        xq += (rt.x_per_route ? r : r / rt.top_k) * ((k / 32) * Q8_1_BYTES);
    }
    int G = 1;   // rows per (virtual) row
    if constexpr (ROUTES) G = rt.pack > 1 ? rt.pack : 1;
    const int64_t nv = n / G, kv = k * G, rbv = rb * G;
    constexpr int V = R * M;
    static_assert(V * TG <= 32 && (V & (V - 1)) == 0, "R*M must be a power of two <= 32/TG");
    __shared__ float red[2][MAXT / 32][TG * V];
    __shared__ uint4 stage[PT::STAGED ? MAXT / 32 : 1][PT::STAGE_CHUNKS];   // warp buffers of staged pieces
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    const int tg = tid % TG;
    const int64_t piece = tid / TG;
    const int64_t P = (kv + PT::VALUES - 1) / PT::VALUES;   // a last partial piece (Q4_0) counts
    const int64_t Pr = (k + PT::VALUES - 1) / PT::VALUES;   // pieces of one real row
    const bool valid = piece < P;
    const typename PT::Pos pos = [&] {
        if constexpr (PT::STAGED) return PT::template pos<TG>(piece, tg, kv);   // lanes past the row still copy their share
        else return PT::pos(valid ? piece : 0);
    }();
    // the piece's place in its real row, which locates its activations
    const typename PT::Pos posr = [&] {
        if (G == 1) return pos;
        if constexpr (PT::STAGED) return PT::template pos<TG>(piece % Pr, tg, k);
        else return PT::pos(piece % Pr);
    }();
    const int64_t stride = (int64_t)gridDim.x * R;
    int64_t n0 = (int64_t)blockIdx.x * R;

    typename PT::W wa[R], wb[R];
    auto load_rows = [&](typename PT::W (&dst)[R], int64_t base) {
        if (!valid && !PT::STAGED) return;
        if constexpr (!MULTI) {
#pragma unroll
            for (int r = 0; r < R; r++) PT::load(dst[r], w0 + (base + r < nv ? base + r : nv - 1) * rbv, pos);
        } else {
            // one lookup per group; a group that crosses a segment end (or the
            // last row) takes the per-row lookup
            const int sgi = seg_index(sg, base);
            if (base + R <= sg.end[sgi]) {
                const uint8_t *row0 = sg.w[sgi] + (base - (sgi ? sg.end[sgi - 1] : 0)) * rb;
#pragma unroll
                for (int r = 0; r < R; r++) PT::load(dst[r], row0 + r * rb, pos);
            } else {
#pragma unroll
                for (int r = 0; r < R; r++) PT::load(dst[r], seg_row(sg, base + r < n ? base + r : n - 1, rb), pos);
            }
        }
    };
    auto store_row = [&](int tok, int64_t r, float v) {
        if constexpr (!MULTI) store_out(y0, yt, (int64_t)tok * ldy0 + r, v);
        else seg_store(sg, yt, tok, r, v);
    };
    // weights never change: the first rows are requested before waiting for
    // the kernel that wrote the activations
    if (n0 < nv) load_rows(wa, n0);
    if constexpr (!ROUTES) mmvq_pdl_enter(sg.chain);
    else asm volatile("griddepcontrol.launch_dependents;" ::: "memory");   // routes waited above

    typename PT::template A<M> act;
    const int m_mine = m_act - tg * M;  // tokens of this thread (may be <= 0)
    PT::template load_act<M>(act, xq + (int64_t)tg * M * ((k / 32) * Q8_1_BYTES), (k / 32) * Q8_1_BYTES,
                             m_mine, posr, valid);

    int buf = 0;
    auto process = [&](const typename PT::W (&cur)[R], int64_t r0) {
        float part[V];
#pragma unroll
        for (int i = 0; i < V; i++) part[i] = 0.0f;
        if constexpr (PT::STAGED) {
#pragma unroll
            for (int r = 0; r < R; r++) {
                typename PT::Wf f;
                PT::prepare(cur[r], pos, stage[warp], f);   // every lane of the warp takes part
                if (valid) {
                    float acc[M];
#pragma unroll
                    for (int mm = 0; mm < M; mm++) acc[mm] = 0.0f;
                    PT::template dot<M>(f, act, pos, acc);
#pragma unroll
                    for (int mm = 0; mm < M; mm++) part[r * M + mm] = acc[mm];
                }
            }
        } else if (valid) {
#pragma unroll
            for (int r = 0; r < R; r++) {
                float acc[M];
#pragma unroll
                for (int mm = 0; mm < M; mm++) acc[mm] = 0.0f;
                PT::template dot<M>(cur[r], act, pos, acc);
#pragma unroll
                for (int mm = 0; mm < M; mm++) part[r * M + mm] = acc[mm];
            }
        }
        if constexpr (ROUTES) {
            if (G > 1) {   // lanes [l - l % Pr, +Pr) hold the pieces of real row (r0 + r) * G + l / Pr
#pragma unroll
                for (int r = 0; r < R; r++) {
                    float v = part[r];
                    for (int o = (int)Pr / 2; o >= 1; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                    if (lane % Pr == 0 && r0 + r < nv) store_row(0, (r0 + r) * G + lane / Pr, v);
                }
                return;
            }
        }
        int idx;
        const float tot = butterfly_tg<V, TG>(part, lane, idx);
        const bool writer = butterfly_writer<V, TG>(lane);
        if (nw == 1) {
            if (writer) {
                const int r = idx / M, tok = tg * M + idx % M;
                if (r0 + r < nv && tok < m_act) store_row(tok, r0 + r, tot);
            }
        } else {
            if (writer) red[buf][warp][tg * V + idx] = tot;
            __syncthreads();
            if (tid < TG * V) {
                float sum = 0.0f;
                for (int j = 0; j < nw; j++) sum += red[buf][j][tid];
                const int g = tid / V, i = tid % V, r = i / M, tok = g * M + i % M;
                if (r0 + r < nv && tok < m_act) store_row(tok, r0 + r, sum);
            }
            buf ^= 1;
        }
    };
    // two register sets in turn: the next rows load while the current compute
    while (n0 < nv) {
        if (n0 + stride < nv) load_rows(wb, n0 + stride);
        process(wa, n0);
        n0 += stride;
        if (n0 >= nv) break;
        if (n0 + stride < nv) load_rows(wa, n0 + stride);
        process(wb, n0);
        n0 += stride;
    }
}

template <class PT, int M, int TG, int R, int MAXT>
inline cudaError_t launch_mmvq_cfg(const MmvqSegs &sg, int64_t k, int64_t rb, const uint8_t *xq, int64_t m, int yt,
                                   cudaStream_t s) {
    const int64_t n = sg.rows();
    const int64_t P = (k + PT::VALUES - 1) / PT::VALUES;
    const int nthr = (int)((P * TG + 31) / 32 * 32);
    if (nthr > MAXT) return cudaErrorInvalidValue;
    auto kern = sg.nseg > 1 ? mmvq_kernel<PT, M, TG, R, MAXT, true> : mmvq_kernel<PT, M, TG, R, MAXT, false>;
    cudaError_t e = cudaSuccess;
    const int per_sm = kernel_occupancy(reinterpret_cast<const void *>(kern), nthr, 0, &e);
    if (per_sm == 0) return e;
    const int64_t groups = (n + R - 1) / R;
    int64_t grid = (int64_t)device_info().sm_count * per_sm;
    if (grid > groups) grid = groups;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)nthr);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, sg, k, rb, xq, (int)m, yt, MmvqRoutes{});
}

// the route-batched launch: CTAs of one route over its rows (two per group),
// as many per route as fill the GPU once.  Rows of at most 32 pieces (one
// warp; MoE down rows of 512 values have 8) take a one-warp instance whose
// buffers are sized for one warp, with registers for 16 resident CTAs per SM
// (4 warps per SM sub-partition: up to 128 registers; only the Q6_K instance
// spills, 40 bytes), and rows of 32 / G whole pieces are packed G to a
// warp-row (rt.pack).  Measured on GB300 against 12 CTAs per SM (168
// registers, no spills) for the E=256 top-8 expert block: 16 tokens 101 ->
// 84 us, 256 tokens 1160 -> 910 us, 4 tokens 37.5 -> 39.6 us.
template <class PT>
inline cudaError_t launch_mmvq_routes_pt(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k,
                                         int64_t rb, const uint8_t *xq, int64_t routes, float *z, cudaStream_t s) {
    if (routes <= 0 || n <= 0) return cudaSuccess;
    const int64_t P = (k + PT::VALUES - 1) / PT::VALUES;
    if (P > 256 || routes > 65535) return cudaErrorInvalidValue;
    const int nthr = (int)((P + 31) / 32 * 32);
    const bool one_warp = nthr == 32;
    constexpr int R = 2;
    // rows of 32 / G whole pieces: G rows per warp-row (all 32 lanes busy)
    MmvqRoutes rtp = rt;
    rtp.pack = 1;
    if (one_warp && k % PT::VALUES == 0 && P <= 16 && 32 % P == 0 && n % (32 / P) == 0) rtp.pack = (int)(32 / P);
    auto kern = one_warp ? mmvq_kernel<PT, 1, 1, 2, 32, false, true> : mmvq_kernel<PT, 1, 1, 2, 256, false, true>;
    cudaError_t e = cudaSuccess;
    const int per_sm = kernel_occupancy(reinterpret_cast<const void *>(kern), nthr, 0, &e);
    if (per_sm == 0) return e;
    const int64_t groups = (n / rtp.pack + R - 1) / R;
    int64_t bx = ((int64_t)device_info().sm_count * per_sm + routes - 1) / routes;
    if (bx > groups) bx = groups;
    if (bx < 1) bx = 1;
    const MmvqSegs sg = mmvq_one_segment(bank, n, z, n);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)bx, (unsigned)routes);
    cfg.blockDim = dim3((unsigned)nthr);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, sg, k, rb, xq, 1, (int)GGUF_F32, rtp);
}

// Configuration by token count (measured on GB300, Q4_K / Q6_K rows of 3072 ..
// 8192 values): up to 4 tokens per thread with the next R rows prefetched
// (R = 4 for 2..4 tokens of Q4_K rows and 2 tokens of Q6_K rows);
// 5..8 tokens either as two threads per piece with 4 tokens each (Q4_K; Q6_K
// and Q8_0 on small matrices) or 8 tokens per thread.  Rows of more than 256
// pieces (32-value pieces of K > 8192) use 512-thread CTAs.
struct MmvqTune {
    bool r4_m1;        // M = 1: R = 4 instead of 2
    bool r8_m1;        // M = 1: R = 8 (overrides r4_m1)
    bool r1_m1;        // M = 1: R = 1 (overrides r4_m1)
    bool tg2_m8;       // 5..8 tokens: two threads per piece
    bool r4_m2;        // 2 tokens: R = 4 instead of 2
    bool r4_m4;        // 3..4 tokens: R = 4 instead of 2
};

template <class PT>
inline cudaError_t launch_mmvq_pt(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s,
                                  int64_t rb, MmvqTune t) {
    const int64_t P = (k + PT::VALUES - 1) / PT::VALUES;
    if (P <= 256) {
        if (m <= 1) {
            if (t.r1_m1) return launch_mmvq_cfg<PT, 1, 1, 1, 256>(sg, k, rb, xq, m, yt, s);
            if (t.r8_m1) return launch_mmvq_cfg<PT, 1, 1, 8, 256>(sg, k, rb, xq, m, yt, s);
            if (t.r4_m1) return launch_mmvq_cfg<PT, 1, 1, 4, 256>(sg, k, rb, xq, m, yt, s);
            return launch_mmvq_cfg<PT, 1, 1, 2, 256>(sg, k, rb, xq, m, yt, s);
        }
        if (m <= 2) {
            if (t.r4_m2) return launch_mmvq_cfg<PT, 2, 1, 4, 256>(sg, k, rb, xq, m, yt, s);
            return launch_mmvq_cfg<PT, 2, 1, 2, 256>(sg, k, rb, xq, m, yt, s);
        }
        if (m <= 4) {
            if (t.r4_m4) return launch_mmvq_cfg<PT, 4, 1, 4, 256>(sg, k, rb, xq, m, yt, s);
            return launch_mmvq_cfg<PT, 4, 1, 2, 256>(sg, k, rb, xq, m, yt, s);
        }
        if (t.tg2_m8 && P <= 128) return launch_mmvq_cfg<PT, 4, 2, 2, 256>(sg, k, rb, xq, m, yt, s);
        return launch_mmvq_cfg<PT, 8, 1, 1, 256>(sg, k, rb, xq, m, yt, s);
    }
    if constexpr (PT::VALUES == 32) {
        if (m <= 1) return launch_mmvq_cfg<PT, 1, 1, 2, 512>(sg, k, rb, xq, m, yt, s);
        if (m <= 2) return launch_mmvq_cfg<PT, 2, 1, 2, 512>(sg, k, rb, xq, m, yt, s);
        if (m <= 4) return launch_mmvq_cfg<PT, 4, 1, 1, 512>(sg, k, rb, xq, m, yt, s);
        return launch_mmvq_cfg<PT, 8, 1, 1, 512>(sg, k, rb, xq, m, yt, s);
    }
    return cudaErrorInvalidValue;  // 64-value pieces: K <= 16384 gives at most 256 pieces
}

cudaError_t launch_mmvq_q8_0(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s);
cudaError_t launch_mmvq_q4_k(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s);
cudaError_t launch_mmvq_q6_k(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s);
cudaError_t launch_mmvq_q4_0(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s);
cudaError_t launch_mmvq_q5_k(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s);
cudaError_t launch_mmvq_mxfp4(const MmvqSegs &sg, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s);
cudaError_t launch_mmvq_routes_q8_0(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s);
cudaError_t launch_mmvq_routes_q4_k(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s);
cudaError_t launch_mmvq_routes_q6_k(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s);
cudaError_t launch_mmvq_routes_q4_0(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s);
cudaError_t launch_mmvq_routes_q5_k(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k, const uint8_t *xq,
                                    int64_t routes, float *z, cudaStream_t s);
cudaError_t launch_mmvq_routes_mxfp4(const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k,
                                     const uint8_t *xq, int64_t routes, float *z, cudaStream_t s);

}  // namespace gg
