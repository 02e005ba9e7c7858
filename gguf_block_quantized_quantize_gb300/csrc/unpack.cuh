// Weight unpack for the tensor-core GEMM: packed Q4_K / Q5_K / Q6_K / Q8_0 /
// Q4_0 / MXFP4 bytes of a
// weight row -> fp16 operand values (each the exact fp32 value of the block
// formula rounded once, or packed-half math where the product is rounded to a
// 16-bit output anyway), stored as 16-byte chunks of a 128-byte-swizzled
// K-major operand tile.
//
// Unit of work ("task"): one weight row, one 64-value K-step, one of PARTS
// parts of it (halves for Q4_K and Q8_0, quarters for Q6_K); a task yields
// CHUNKS 8-value chunks (16-byte fp16 chunks of the swizzled row), chunk e of
// part j at position chunk(j, e) of the row.  (Halves for Q4_K, Q5_K, Q8_0,
// Q4_0 and MXFP4.)  Consecutive lanes take the parts
// of one row, so a warp-wide load reads contiguous bytes of 16 (8) rows, and
// every packed byte is read once.
#pragma once

#include "common.cuh"

namespace gg {

// ---------------------------------------------------------------- packed-byte helpers

// exact small integer -> float: 2^23 + byte, then subtract
__device__ __forceinline__ float byte_to_f(uint32_t word, int byte, float bias) {
    const uint32_t sel = (uint32_t)byte | (4u << 4) | (4u << 8) | (7u << 12);
    return __uint_as_float(__byte_perm(word, 0x4B000000u, sel)) + bias;
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// ---------------------------------------------------------------- quarter tasks

// (1024 + byte) as fp16 for bytes 2i and 2i+1 of w (i = 0, 1)
__device__ __forceinline__ uint32_t bytes_to_h2_1024(uint32_t w, int i) {
    return __byte_perm(w, 0x64646464u, i == 0 ? 0x4140u : 0x4342u);
}
__device__ __forceinline__ __half2 u32_as_h2(uint32_t v) { return *reinterpret_cast<const __half2 *>(&v); }
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<const uint32_t *>(&h); }

template <int WT>
struct KQ;

// Q4_K: K-step ks is chunk c = ks % 4 of super-block ks / 4 (values 64c ..
// 64c + 63); half j holds quant bytes [32c + 16j, +16), whose low nibbles are
// values 16j .. 16j+15 of sub-block 2c (chunks 2j, 2j+1) and whose high
// nibbles are the same values of sub-block 2c + 1 (chunks 4 + 2j, 5 + 2j).
template <>
struct KQ<GGUF_Q4_K> {
    static constexpr int PARTS = 2, CHUNKS = 4;
    static __device__ __forceinline__ int chunk(int j, int e) { return e < 2 ? 2 * j + e : 2 + 2 * j + e; }
    uint4 hdr, q;
    __device__ __forceinline__ void load(const uint8_t *row, int ks, int j, int64_t) {
        const uint8_t *blk = row + (int64_t)(ks >> 2) * Q4_K_BYTES;
        hdr = *reinterpret_cast<const uint4 *>(blk);
        q = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * (ks & 3) + 16 * j);
    }
    // a * q - b with a = d * s, b = dmin * m (both exact in fp32) for the two sub-blocks
    __device__ __forceinline__ void scales(int ks, float &a0, float &b0, float &a1, float &b1) const {
        const uint32_t sc[3] = {hdr.y, hdr.z, hdr.w};
        const float d = h2f(hdr.x & 0xffff), dmin = h2f(hdr.x >> 16);
        int s, m;
        q4k_scale_min(sc, 2 * (ks & 3), s, m);
        a0 = __fmul_rn(d, (float)s);
        b0 = __fmul_rn(dmin, (float)m);
        q4k_scale_min(sc, 2 * (ks & 3) + 1, s, m);
        a1 = __fmul_rn(d, (float)s);
        b1 = __fmul_rn(dmin, (float)m);
    }
    __device__ __forceinline__ void unpack_f32(int ks, float (&v)[32]) const {
        float a0, b0, a1, b1;
        scales(ks, a0, b0, a1, b1);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int h = 0; h < 4; h++) {
            const uint32_t lo = w[h] & 0x0F0F0F0Fu, hi = (w[h] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
            for (int b = 0; b < 4; b++) {
                v[4 * h + b] = fmaf(a0, byte_to_f(lo, b, -8388608.0f), -b0);   // a * q exact, one rounding
                v[16 + 4 * h + b] = fmaf(a1, byte_to_f(hi, b, -8388608.0f), -b1);
            }
        }
    }
    __device__ __forceinline__ void unpack_h2(int ks, uint32_t (&out)[16]) const {
        float a0, b0, a1, b1;
        scales(ks, a0, b0, a1, b1);
        const __half2 a02 = __float2half2_rn(a0), nb02 = __float2half2_rn(-b0);
        const __half2 a12 = __float2half2_rn(a1), nb12 = __float2half2_rn(-b1);
        const __half2 k1024 = __float2half2_rn(1024.0f);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int h = 0; h < 4; h++) {
            const uint32_t lo = w[h] & 0x0F0F0F0Fu, hi = (w[h] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
            for (int p = 0; p < 2; p++) {
                out[2 * h + p] = h2_as_u32(__hfma2(__hsub2(u32_as_h2(bytes_to_h2_1024(lo, p)), k1024), a02, nb02));
                out[8 + 2 * h + p] = h2_as_u32(__hfma2(__hsub2(u32_as_h2(bytes_to_h2_1024(hi, p)), k1024), a12, nb12));
            }
        }
    }
};

// Q6_K: K-step ks is half h = (ks / 2) % 2, nibble jj = ks % 2 of super-block
// ks / 4: values 0..31 of the step are run g = 2jj (l = 0..31), 32..63 run
// g = 2jj + 1.  Quarter i: l = 8i .. 8i+7 of both runs, i.e. ql bytes
// [64h + 8i, +8) (run 2jj) and [64h + 32 + 8i, +8) (run 2jj + 1), nibble jj,
// and qh bytes [32h + 8i, +8), bits 2g; scales sc[8h + 2g + i / 2].
template <>
struct KQ<GGUF_Q6_K> {
    static constexpr int PARTS = 4, CHUNKS = 2;
    static __device__ __forceinline__ int chunk(int i, int e) { return e == 0 ? i : 4 + i; }
    uint32_t qa[2], qb[2], qh[2], sc, dw;
    __device__ __forceinline__ void load(const uint8_t *row, int ks, int i, int64_t) {
        const uint8_t *blk = row + (int64_t)(ks >> 2) * Q6_K_BYTES;
        const int h = (ks >> 1) & 1, jj = ks & 1;
        ldw_a2<2>(blk + 64 * h + 8 * i, qa);
        ldw_a2<2>(blk + 64 * h + 32 + 8 * i, qb);
        ldw_a2<2>(blk + 128 + 32 * h + 8 * i, qh);
        uint32_t s4[1];
        ldw_a2<1>(blk + 192 + 8 * h + 4 * jj, s4);           // sc[8h + 4jj .. +3]
        sc = __byte_perm(s4[0], 0u, (uint32_t)(i >> 1) | ((uint32_t)(2 + (i >> 1)) << 4));
        dw = ld_u16(blk + 208);
    }
    // unsigned 6-bit quants of 4 values of run gg (0: chunk i, 1: chunk 4 + i), word h
    __device__ __forceinline__ uint32_t quants(int ks, int gg, int h) const {
        const int jj = ks & 1;
        const uint32_t ql = gg ? qb[h] : qa[h];
        return ((ql >> (4 * jj)) & 0x0F0F0F0Fu) | (((qh[h] >> (4 * jj + 2 * gg)) & 0x03030303u) << 4);
    }
    __device__ __forceinline__ void dscales(float &ds0, float &ds1) const {
        const float d = h2f((uint16_t)dw);
        ds0 = __fmul_rn(d, (float)(int)(int8_t)(sc & 0xff));
        ds1 = __fmul_rn(d, (float)(int)(int8_t)((sc >> 8) & 0xff));
    }
    // exact fp32 values (d * sc * (q - 32) fits in 24 bits)
    __device__ __forceinline__ void unpack_f32(int ks, float (&v)[16]) const {
        float ds0, ds1;
        dscales(ds0, ds1);
#pragma unroll
        for (int gg = 0; gg < 2; gg++)
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint32_t u = quants(ks, gg, h);
#pragma unroll
                for (int j = 0; j < 4; j++) v[8 * gg + 4 * h + j] = __fmul_rn(gg ? ds1 : ds0, byte_to_f(u, j, -8388640.0f));
            }
    }
    __device__ __forceinline__ void unpack_h2(int ks, uint32_t (&out)[8]) const {
        float ds0, ds1;
        dscales(ds0, ds1);
        const __half2 d0 = __float2half2_rn(ds0), d1 = __float2half2_rn(ds1), k1056 = __float2half2_rn(1056.0f);
#pragma unroll
        for (int gg = 0; gg < 2; gg++)
#pragma unroll
            for (int h = 0; h < 2; h++) {
                const uint32_t u = quants(ks, gg, h);
#pragma unroll
                for (int p = 0; p < 2; p++) {
                    const __half2 qq = __hsub2(u32_as_h2(bytes_to_h2_1024(u, p)), k1056);  // q - 32
                    out[4 * gg + 2 * h + p] = h2_as_u32(__hmul2(qq, gg ? d1 : d0));
                }
            }
    }
};

// Q8_0: K-step ks is blocks 2ks (chunks 0..3) and 2ks + 1 (chunks 4..7, absent
// past the end when K % 64 == 32); half j is block 2ks + j.
template <>
struct KQ<GGUF_Q8_0> {
    static constexpr int PARTS = 2, CHUNKS = 4;
    static __device__ __forceinline__ int chunk(int j, int e) { return 4 * j + e; }
    uint32_t q[8], dw;
    __device__ __forceinline__ void load(const uint8_t *row, int ks, int j, int64_t kblocks) {
        const int64_t b = 2 * (int64_t)ks + j;
        if (b < kblocks) {
            const uint8_t *blk = row + b * Q8_0_BYTES;
            dw = ld_u16(blk);
            ldw_a2<8>(blk + 2, q);
        } else {
            dw = 0u;
#pragma unroll
            for (int i = 0; i < 8; i++) q[i] = 0u;
        }
    }
    __device__ __forceinline__ void unpack_f32(int, float (&v)[32]) const {
        const float d = h2f((uint16_t)dw);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t u = q[i] ^ 0x80808080u;  // signed byte + 128
#pragma unroll
            for (int b = 0; b < 4; b++) v[4 * i + b] = __fmul_rn(d, byte_to_f(u, b, -8388736.0f));
        }
    }
    // d * q is exact in fp32 and rounded once to fp16 either way
    __device__ __forceinline__ void unpack_h2(int, uint32_t (&out)[16]) const {
        const __half2 d2 = __halves2half2(__ushort_as_half((uint16_t)dw), __ushort_as_half((uint16_t)dw));
        const __half2 k1152 = __float2half2_rn(1152.0f);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t u = q[i] ^ 0x80808080u;
#pragma unroll
            for (int p = 0; p < 2; p++)
                out[2 * i + p] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(bytes_to_h2_1024(u, p)), k1152), d2));
        }
    }
};

// Q5_K: as Q4_K (the same header; quant bytes at 48 instead of 16), and half
// j also takes high-bit bytes [16j, +16) (at byte 16 of the block), whose bits
// 2c and 2c + 1 are the fifth bits of the low- and high-nibble sub-blocks.
template <>
struct KQ<GGUF_Q5_K> {
    static constexpr int PARTS = 2, CHUNKS = 4;
    static __device__ __forceinline__ int chunk(int j, int e) { return e < 2 ? 2 * j + e : 2 + 2 * j + e; }
    uint4 hdr, q, qh;
    __device__ __forceinline__ void load(const uint8_t *row, int ks, int j, int64_t) {
        const uint8_t *blk = row + (int64_t)(ks >> 2) * Q5_K_BYTES;
        hdr = *reinterpret_cast<const uint4 *>(blk);
        qh = *reinterpret_cast<const uint4 *>(blk + 16 + 16 * j);
        q = *reinterpret_cast<const uint4 *>(blk + 48 + 32 * (ks & 3) + 16 * j);
    }
    __device__ __forceinline__ void scales(int ks, float &a0, float &b0, float &a1, float &b1) const {
        const uint32_t sc[3] = {hdr.y, hdr.z, hdr.w};
        const float d = h2f(hdr.x & 0xffff), dmin = h2f(hdr.x >> 16);
        int s, m;
        q4k_scale_min(sc, 2 * (ks & 3), s, m);
        a0 = __fmul_rn(d, (float)s);
        b0 = __fmul_rn(dmin, (float)m);
        q4k_scale_min(sc, 2 * (ks & 3) + 1, s, m);
        a1 = __fmul_rn(d, (float)s);
        b1 = __fmul_rn(dmin, (float)m);
    }
    // 5-bit quants of the low / high nibble sub-block, 4 per word
    __device__ __forceinline__ void quants(int ks, int h, uint32_t &lo, uint32_t &hi) const {
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
        const uint32_t b[4] = {qh.x, qh.y, qh.z, qh.w};
        const uint32_t hb = b[h] >> (2 * (ks & 3));
        lo = (w[h] & 0x0F0F0F0Fu) | ((hb << 4) & 0x10101010u);
        hi = ((w[h] >> 4) & 0x0F0F0F0Fu) | ((hb << 3) & 0x10101010u);
    }
    __device__ __forceinline__ void unpack_f32(int ks, float (&v)[32]) const {
        float a0, b0, a1, b1;
        scales(ks, a0, b0, a1, b1);
#pragma unroll
        for (int h = 0; h < 4; h++) {
            uint32_t lo, hi;
            quants(ks, h, lo, hi);
#pragma unroll
            for (int b = 0; b < 4; b++) {
                v[4 * h + b] = fmaf(a0, byte_to_f(lo, b, -8388608.0f), -b0);   // a * q exact, one rounding
                v[16 + 4 * h + b] = fmaf(a1, byte_to_f(hi, b, -8388608.0f), -b1);
            }
        }
    }
    __device__ __forceinline__ void unpack_h2(int ks, uint32_t (&out)[16]) const {
        float a0, b0, a1, b1;
        scales(ks, a0, b0, a1, b1);
        const __half2 a02 = __float2half2_rn(a0), nb02 = __float2half2_rn(-b0);
        const __half2 a12 = __float2half2_rn(a1), nb12 = __float2half2_rn(-b1);
        const __half2 k1024 = __float2half2_rn(1024.0f);
#pragma unroll
        for (int h = 0; h < 4; h++) {
            uint32_t lo, hi;
            quants(ks, h, lo, hi);
#pragma unroll
            for (int p = 0; p < 2; p++) {
                out[2 * h + p] = h2_as_u32(__hfma2(__hsub2(u32_as_h2(bytes_to_h2_1024(lo, p)), k1024), a02, nb02));
                out[8 + 2 * h + p] = h2_as_u32(__hfma2(__hsub2(u32_as_h2(bytes_to_h2_1024(hi, p)), k1024), a12, nb12));
            }
        }
    }
};

// Q4_0: as Q8_0, K-step ks is blocks 2ks (chunks 0..3) and 2ks + 1 (chunks
// 4..7, absent past the end when K % 64 == 32); half j is block 2ks + j, whose
// 16 quant bytes hold values 0..15 in the low nibbles and 16..31 in the high.
template <>
struct KQ<GGUF_Q4_0> {
    static constexpr int PARTS = 2, CHUNKS = 4;
    static __device__ __forceinline__ int chunk(int j, int e) { return 4 * j + e; }
    uint32_t q[4], dw;
    __device__ __forceinline__ void load(const uint8_t *row, int ks, int j, int64_t kblocks) {
        const int64_t b = 2 * (int64_t)ks + j;
        if (b < kblocks) {
            const uint8_t *blk = row + b * Q4_0_BYTES;
            dw = ld_u16(blk);
            ldw_a2<4>(blk + 2, q);
        } else {
            dw = 0u;
#pragma unroll
            for (int i = 0; i < 4; i++) q[i] = 0u;
        }
    }
    // d * (q - 8) is exact in fp32
    __device__ __forceinline__ void unpack_f32(int, float (&v)[32]) const {
        const float d = h2f((uint16_t)dw);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t lo = q[i] & 0x0F0F0F0Fu, hi = (q[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
            for (int b = 0; b < 4; b++) {
                v[4 * i + b] = __fmul_rn(d, byte_to_f(lo, b, -8388616.0f));
                v[16 + 4 * i + b] = __fmul_rn(d, byte_to_f(hi, b, -8388616.0f));
            }
        }
    }
    // q - 8 is exact in fp16 and the product is rounded once, as above
    __device__ __forceinline__ void unpack_h2(int, uint32_t (&out)[16]) const {
        const __half2 d2 = __halves2half2(__ushort_as_half((uint16_t)dw), __ushort_as_half((uint16_t)dw));
        const __half2 k1032 = __float2half2_rn(1032.0f);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const uint32_t lo = q[i] & 0x0F0F0F0Fu, hi = (q[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
            for (int p = 0; p < 2; p++) {
                out[2 * i + p] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(bytes_to_h2_1024(lo, p)), k1032), d2));
                out[8 + 2 * i + p] = h2_as_u32(__hmul2(__hsub2(u32_as_h2(bytes_to_h2_1024(hi, p)), k1032), d2));
            }
        }
    }
};

// MXFP4: as Q4_0, K-step ks is blocks 2ks and 2ks + 1 (absent past the end when
// K % 64 == 32), half j block 2ks + j: 17 bytes at any address, the E8M0
// exponent then the codes of values 0..15 (low nibbles) and 16..31 (high).
template <>
struct KQ<GGUF_MXFP4> {
    static constexpr int PARTS = 2, CHUNKS = 4;
    static __device__ __forceinline__ int chunk(int j, int e) { return 4 * j + e; }
    uint32_t q[4], e;
    __device__ __forceinline__ void load(const uint8_t *row, int ks, int j, int64_t kblocks) {
        const int64_t b = 2 * (int64_t)ks + j;
        if (b < kblocks) {
            ld_mxfp4_block(row + b * MXFP4_BYTES, e, q);
        } else {
            e = 0u;
#pragma unroll
            for (int i = 0; i < 4; i++) q[i] = 0x88888888u;   // code 8: -0
        }
    }
    // 2^(e - 128) * k, exact in fp32 (or inf past its range)
    __device__ __forceinline__ void unpack_f32(int, float (&v)[32]) const {
        const float d = e8m0_half(e);
#pragma unroll
        for (int i = 0; i < 4; i++) {
            // biased bytes of values (4i, 16+4i, 4i+1, 17+4i) and (4i+2, 18+4i, 4i+3, 19+4i)
            const uint32_t u0 = mxfp4_biased4(q[i]), u1 = mxfp4_biased4(q[i] >> 16);
            const uint32_t lo = __byte_perm(u0, u1, 0x6420), hi = __byte_perm(u0, u1, 0x7531);
#pragma unroll
            for (int b = 0; b < 4; b++) {
                v[4 * i + b] = __fmul_rn(d, byte_to_f(lo, b, -8388624.0f));
                v[16 + 4 * i + b] = __fmul_rn(d, byte_to_f(hi, b, -8388624.0f));
            }
        }
    }
    // the block factor can lie outside the fp16 range: round the exact fp32 values once
    __device__ __forceinline__ void unpack_h2(int ks, uint32_t (&out)[16]) const {
        float v[32];
        unpack_f32(ks, v);
#pragma unroll
        for (int i = 0; i < 16; i++) out[i] = pack_h2(v[2 * i], v[2 * i + 1]);
    }
};

// fp32 values -> one fp16 operand (single rounding)
template <int V>
__device__ __forceinline__ void pack_single(const float (&v)[V], uint32_t (&hi)[V / 2]) {
#pragma unroll
    for (int i = 0; i < V / 2; i++) hi[i] = pack_h2(v[2 * i], v[2 * i + 1]);
}
// fp32 values -> hi + lo fp16 operands with hi + lo = v to ~2^-22
template <int V>
__device__ __forceinline__ void pack_split(const float (&v)[V], uint32_t (&hi)[V / 2], uint32_t (&lo)[V / 2]) {
#pragma unroll
    for (int i = 0; i < V / 2; i++) {
        const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        const float2 hf = __half22float2(h);
        hi[i] = h2_as_u32(h);
        lo[i] = pack_h2(v[2 * i] - hf.x, v[2 * i + 1] - hf.y);
    }
}

// store the chunks of task part j into row `row` of a 128-byte-swizzled tile
template <class U>
__device__ __forceinline__ void store_sw128_task(uint8_t *tile, int row, int j, const uint32_t (&v)[4 * U::CHUNKS]) {
    uint8_t *base = tile + row * 128;
#pragma unroll
    for (int e = 0; e < U::CHUNKS; e++)
        *reinterpret_cast<uint4 *>(base + ((U::chunk(j, e) ^ (row & 7)) * 16)) =
            make_uint4(v[4 * e], v[4 * e + 1], v[4 * e + 2], v[4 * e + 3]);
}

}  // namespace gg
