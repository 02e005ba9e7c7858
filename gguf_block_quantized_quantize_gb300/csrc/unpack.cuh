// Weight unpack for the tensor-core kernels: packed Q4_K / Q6_K / Q8_0 bytes of
// one weight row and one 64-value K-step -> 64 fp16 values (each the exact fp32
// value of the block formula rounded once), stored as one 128-byte row of a
// 128-byte-swizzled K-major operand tile.
#pragma once

#include "common.cuh"

namespace gg {

// ---------------------------------------------------------------- packed-byte loads

// Exactly the 4*N bytes at the 2-byte-aligned p, as N words; reads only
// [p - 2, p + 4N) (aligned words, the last two bytes by a 16-bit load).
template <int N>
__device__ __forceinline__ void ldw_a2(const uint8_t *p, uint32_t (&o)[N]) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    if ((a & 2) == 0) {
#pragma unroll
        for (int i = 0; i < N; i++) o[i] = ld_u32(p + 4 * i);
    } else {
        const uint8_t *b = p - 2;
        uint32_t w[N + 1];
#pragma unroll
        for (int i = 0; i < N; i++) w[i] = ld_u32(b + 4 * i);
        w[N] = ld_u16(b + 4 * N);
#pragma unroll
        for (int i = 0; i < N; i++) o[i] = __funnelshift_r(w[i], w[i + 1], 16);
    }
}

// exact small integer -> float: 2^23 + byte, then subtract
__device__ __forceinline__ float byte_to_f(uint32_t word, int byte, float bias) {
    const uint32_t sel = (uint32_t)byte | (4u << 4) | (4u << 8) | (7u << 12);
    return __uint_as_float(__byte_perm(word, 0x4B000000u, sel)) + bias;
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// ---------------------------------------------------------------- per-type K-step units

// Packed bytes of one weight row for one K-step of 64 values.
template <int WT>
struct KUnit;

template <>
struct KUnit<GGUF_Q4_K> {
    uint4 hdr, q0, q1;
    __device__ __forceinline__ void load(const uint8_t *row, int ks) {
        const uint8_t *blk = row + (int64_t)(ks >> 2) * Q4_K_BYTES;
        const int c = ks & 3;
        hdr = *reinterpret_cast<const uint4 *>(blk);
        q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
        q1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
    }
    // 64 values: [0, 32) = low nibbles of the 32 quant bytes (sub-block 2c),
    // [32, 64) = high nibbles (sub-block 2c + 1); v = (d*s)*q - dmin*m.
    __device__ __forceinline__ void unpack(int ks, uint32_t (&out)[32]) const {
        const int c = ks & 3;
        const uint32_t sc[3] = {hdr.y, hdr.z, hdr.w};
        const float d = h2f(hdr.x & 0xffff), dmin = h2f(hdr.x >> 16);
        int s0, m0, s1, m1;
        q4k_scale_min(sc, 2 * c, s0, m0);
        q4k_scale_min(sc, 2 * c + 1, s1, m1);
        const float a0 = __fmul_rn(d, (float)s0), b0 = __fmul_rn(dmin, (float)m0);
        const float a1 = __fmul_rn(d, (float)s1), b1 = __fmul_rn(dmin, (float)m1);
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
            float v[4], u[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                v[j] = fmaf(a0, byte_to_f(lo, j, -8388608.0f), -b0);
                u[j] = fmaf(a1, byte_to_f(hi, j, -8388608.0f), -b1);
            }
            out[2 * i] = pack_h2(v[0], v[1]);
            out[2 * i + 1] = pack_h2(v[2], v[3]);
            out[16 + 2 * i] = pack_h2(u[0], u[1]);
            out[16 + 2 * i + 1] = pack_h2(u[2], u[3]);
        }
    }
};

template <>
struct KUnit<GGUF_Q6_K> {
    uint32_t ql[16], qh[8], sc, dw;
    // K-step ks: super-block ks/4, half h = (ks%4)/2, quarter j = ks%2 -> the
    // runs g = 2j, 2j+1 of the half; needs the half's 64 ql and 32 qh bytes.
    __device__ __forceinline__ void load(const uint8_t *row, int ks) {
        const uint8_t *blk = row + (int64_t)(ks >> 2) * Q6_K_BYTES;
        const int h = (ks >> 1) & 1, j = ks & 1;
        ldw_a2<16>(blk + 64 * h, ql);
        ldw_a2<8>(blk + 128 + 32 * h, qh);
        uint32_t s[1];
        ldw_a2<1>(blk + 192 + 8 * h + 4 * j, s);
        sc = s[0];
        dw = ld_u16(blk + 208);
    }
    // values [32gg, 32gg + 32) = run g = 2j + gg: low 4 bits from ql byte
    // 32*gg + l (nibble j), high 2 bits from qh byte l (bits 2g, 2g+1);
    // v = (d*sc) * (q - 32), scale sc[8h + 2g + l/16].
    __device__ __forceinline__ void unpack(int ks, uint32_t (&out)[32]) const {
        const int j = ks & 1;
        const float d = h2f(dw & 0xffff);
#pragma unroll
        for (int gg = 0; gg < 2; gg++) {
            const float ds0 = __fmul_rn(d, (float)(int)(int8_t)((sc >> (16 * gg)) & 0xff));
            const float ds1 = __fmul_rn(d, (float)(int)(int8_t)((sc >> (16 * gg + 8)) & 0xff));
            const int hshift = 4 * j + 2 * gg;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const uint32_t q4 = ((ql[8 * gg + i] >> (4 * j)) & 0x0F0F0F0Fu) |
                                    (((qh[i] >> hshift) & 0x03030303u) << 4);
                const float dsc = i < 4 ? ds0 : ds1;  // values l = 4i .. 4i+3: l < 16 uses the first scale
                float v[4];
#pragma unroll
                for (int t = 0; t < 4; t++) v[t] = __fmul_rn(dsc, byte_to_f(q4, t, -8388640.0f));
                out[16 * gg + 2 * i] = pack_h2(v[0], v[1]);
                out[16 * gg + 2 * i + 1] = pack_h2(v[2], v[3]);
            }
        }
    }
};

template <>
struct KUnit<GGUF_Q8_0> {
    uint32_t q[2][8];
    uint32_t d2;
    int nblk;  // 2, or 1 for a trailing half step when k % 64 == 32
    int64_t kblocks;
    __device__ __forceinline__ void load(const uint8_t *row, int ks) {
        const int64_t b0 = 2 * (int64_t)ks;
        nblk = (b0 + 1 < kblocks) ? 2 : 1;
        d2 = 0;
#pragma unroll
        for (int t = 0; t < 2; t++) {
            if (t < nblk) {
                const uint8_t *blk = row + (b0 + t) * Q8_0_BYTES;
                d2 |= (uint32_t)ld_u16(blk) << (16 * t);
                ldw_a2<8>(blk + 2, q[t]);
            } else {
#pragma unroll
                for (int i = 0; i < 8; i++) q[t][i] = 0u;  // the missing block decodes with d = 0 below
            }
        }
    }
    __device__ __forceinline__ void unpack(int, uint32_t (&out)[32]) const {
#pragma unroll
        for (int t = 0; t < 2; t++) {
            const float d = t < nblk ? h2f((d2 >> (16 * t)) & 0xffff) : 0.0f;
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const uint32_t u = q[t][i] ^ 0x80808080u;  // signed byte + 128
                float v[4];
#pragma unroll
                for (int b = 0; b < 4; b++) v[b] = __fmul_rn(d, byte_to_f(u, b, -8388736.0f));
                out[16 * t + 2 * i] = pack_h2(v[0], v[1]);
                out[16 * t + 2 * i + 1] = pack_h2(v[2], v[3]);
            }
        }
    }
};

// store 64 fp16 (32 words) as one 128-byte row of a 128-byte-swizzled tile
__device__ __forceinline__ void store_sw128_row(uint8_t *tile, int row, const uint32_t (&v)[32]) {
    uint8_t *base = tile + row * 128;
#pragma unroll
    for (int c = 0; c < 8; c++) {
        const int pc = c ^ (row & 7);
        *reinterpret_cast<uint4 *>(base + pc * 16) = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    }
}

}  // namespace gg

namespace gg {

// ---------------------------------------------------------------- half-row units
//
// A K-step of 64 values of one weight row, split in two halves of 32 values
// (one 32-value sub-block, or two 16-value Q6_K sub-blocks, or one Q8_0
// block), each produced by its own thread.  `H2` selects packed-half math
// (two fp16 roundings per value instead of one; used when the product is
// rounded to a 16-bit output anyway).

// (1024 + byte) as fp16 for bytes 2i and 2i+1 of w (i = 0, 1)
__device__ __forceinline__ uint32_t bytes_to_h2_1024(uint32_t w, int i) {
    return __byte_perm(w, 0x64646464u, i == 0 ? 0x4140u : 0x4342u);
}
__device__ __forceinline__ __half2 u32_as_h2(uint32_t v) { return *reinterpret_cast<const __half2 *>(&v); }
__device__ __forceinline__ uint32_t h2_as_u32(__half2 h) { return *reinterpret_cast<const uint32_t *>(&h); }

template <int WT>
struct KHalf;

template <>
struct KHalf<GGUF_Q4_K> {
    uint4 hdr, q0, q1;
    __device__ __forceinline__ void load(const uint8_t *row, int ks, int) {
        const uint8_t *blk = row + (int64_t)(ks >> 2) * Q4_K_BYTES;
        const int c = ks & 3;
        hdr = *reinterpret_cast<const uint4 *>(blk);
        q0 = *reinterpret_cast<const uint4 *>(blk + 16 + 32 * c);
        q1 = *reinterpret_cast<const uint4 *>(blk + 32 + 32 * c);
    }
    // half 0: low nibbles (sub-block 2c), half 1: high nibbles (sub-block 2c+1)
    __device__ __forceinline__ void scales(int ks, int half, float &a, float &b) const {
        const uint32_t sc[3] = {hdr.y, hdr.z, hdr.w};
        int s, m;
        q4k_scale_min(sc, 2 * (ks & 3) + half, s, m);
        a = __fmul_rn(h2f(hdr.x & 0xffff), (float)s);
        b = __fmul_rn(h2f(hdr.x >> 16), (float)m);
    }
    __device__ __forceinline__ uint32_t nibbles(int i, int half) const {
        const uint32_t w[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        return half ? ((w[i] >> 4) & 0x0F0F0F0Fu) : (w[i] & 0x0F0F0F0Fu);
    }
    // exact fp32 block values (a*q is exact; the subtraction rounds once)
    __device__ __forceinline__ void unpack_f32(int ks, int half, float (&v)[32]) const {
        float a, b;
        scales(ks, half, a, b);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t nib = nibbles(i, half);
#pragma unroll
            for (int j = 0; j < 4; j++) v[4 * i + j] = fmaf(a, byte_to_f(nib, j, -8388608.0f), -b);
        }
    }
    __device__ __forceinline__ void unpack_h2(int ks, int half, uint32_t (&out)[16]) const {
        float a, b;
        scales(ks, half, a, b);
        const __half2 a2 = __float2half2_rn(a), nb2 = __float2half2_rn(-b), k1024 = __float2half2_rn(1024.0f);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t nib = nibbles(i, half);
#pragma unroll
            for (int p = 0; p < 2; p++) {
                const __half2 q = __hsub2(u32_as_h2(bytes_to_h2_1024(nib, p)), k1024);
                out[2 * i + p] = h2_as_u32(__hfma2(q, a2, nb2));
            }
        }
    }
};

template <>
struct KHalf<GGUF_Q6_K> {
    uint32_t ql[8], qh[8], sc, dw;
    // K-step ks: super-block ks/4, half h = (ks%4)/2, j = ks%2; this thread's
    // half gg is run g = 2j + gg: ql bytes [64h + 32gg, +32), nibble j.
    __device__ __forceinline__ void load(const uint8_t *row, int ks, int gg) {
        const uint8_t *blk = row + (int64_t)(ks >> 2) * Q6_K_BYTES;
        const int h = (ks >> 1) & 1, j = ks & 1;
        ldw_a2<8>(blk + 64 * h + 32 * gg, ql);
        ldw_a2<8>(blk + 128 + 32 * h, qh);
        sc = ld_u16(blk + 192 + 8 * h + 2 * (2 * j + gg));   // scales of l < 16 and l >= 16
        dw = ld_u16(blk + 208);
    }
    __device__ __forceinline__ uint32_t quants(int ks, int gg, int i) const {
        const int j = ks & 1;
        return ((ql[i] >> (4 * j)) & 0x0F0F0F0Fu) | (((qh[i] >> (4 * j + 2 * gg)) & 0x03030303u) << 4);
    }
    __device__ __forceinline__ void dscales(float &ds0, float &ds1) const {
        const float d = h2f(dw & 0xffff);
        ds0 = __fmul_rn(d, (float)(int)(int8_t)(sc & 0xff));
        ds1 = __fmul_rn(d, (float)(int)(int8_t)((sc >> 8) & 0xff));
    }
    // exact fp32 values (d*sc*(q-32) fits in 24 bits)
    __device__ __forceinline__ void unpack_f32(int ks, int gg, float (&v)[32]) const {
        float ds0, ds1;
        dscales(ds0, ds1);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t q4 = quants(ks, gg, i);
#pragma unroll
            for (int t = 0; t < 4; t++) v[4 * i + t] = __fmul_rn(i < 4 ? ds0 : ds1, byte_to_f(q4, t, -8388640.0f));
        }
    }
    __device__ __forceinline__ void unpack_h2(int ks, int gg, uint32_t (&out)[16]) const {
        float ds0, ds1;
        dscales(ds0, ds1);
        const __half2 d0 = __float2half2_rn(ds0), d1 = __float2half2_rn(ds1), k1056 = __float2half2_rn(1056.0f);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t q4 = quants(ks, gg, i);
#pragma unroll
            for (int p = 0; p < 2; p++) {
                const __half2 q = __hsub2(u32_as_h2(bytes_to_h2_1024(q4, p)), k1056);  // q - 32
                out[2 * i + p] = h2_as_u32(__hmul2(q, i < 4 ? d0 : d1));
            }
        }
    }
};

template <>
struct KHalf<GGUF_Q8_0> {
    uint32_t q[8];
    uint32_t dw;
    int64_t kblocks;
    // half t of K-step ks is block 2*ks + t (absent past the end when k % 64 == 32)
    __device__ __forceinline__ void load(const uint8_t *row, int ks, int t) {
        const int64_t b = 2 * (int64_t)ks + t;
        if (b < kblocks) {
            const uint8_t *blk = row + b * Q8_0_BYTES;
            dw = ld_u16(blk);
            ldw_a2<8>(blk + 2, q);
        } else {
            dw = 0;
#pragma unroll
            for (int i = 0; i < 8; i++) q[i] = 0u;
        }
    }
    __device__ __forceinline__ void unpack_f32(int, int, float (&v)[32]) const {
        const float d = h2f((uint16_t)dw);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t u = q[i] ^ 0x80808080u;  // signed byte + 128
#pragma unroll
            for (int b = 0; b < 4; b++) v[4 * i + b] = __fmul_rn(d, byte_to_f(u, b, -8388736.0f));
        }
    }
    // d * q is exact in fp32 and rounded once to fp16 either way
    __device__ __forceinline__ void unpack_h2(int, int, uint32_t (&out)[16]) const {
        const __half2 d2 = __halves2half2(__ushort_as_half((uint16_t)dw), __ushort_as_half((uint16_t)dw));
        const __half2 k1152 = __float2half2_rn(1152.0f);
#pragma unroll
        for (int i = 0; i < 8; i++) {
            const uint32_t u = q[i] ^ 0x80808080u;
#pragma unroll
            for (int p = 0; p < 2; p++) {
                const __half2 qq = __hsub2(u32_as_h2(bytes_to_h2_1024(u, p)), k1152);
                out[2 * i + p] = h2_as_u32(__hmul2(qq, d2));
            }
        }
    }
};

// fp32 values -> one fp16 operand (single rounding)
__device__ __forceinline__ void pack_single(const float (&v)[32], uint32_t (&hi)[16]) {
#pragma unroll
    for (int i = 0; i < 16; i++) hi[i] = pack_h2(v[2 * i], v[2 * i + 1]);
}
// fp32 values -> hi + lo fp16 operands with hi + lo = v to ~2^-22
__device__ __forceinline__ void pack_split(const float (&v)[32], uint32_t (&hi)[16], uint32_t (&lo)[16]) {
#pragma unroll
    for (int i = 0; i < 16; i++) {
        const __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
        const float2 hf = __half22float2(h);
        hi[i] = h2_as_u32(h);
        lo[i] = pack_h2(v[2 * i] - hf.x, v[2 * i + 1] - hf.y);
    }
}

// store 32 fp16 (16 words) as chunks [4*half, 4*half + 4) of a 128-byte swizzled row
__device__ __forceinline__ void store_sw128_half(uint8_t *tile, int row, int half, const uint32_t (&v)[16]) {
    uint8_t *base = tile + row * 128;
#pragma unroll
    for (int c = 0; c < 4; c++) {
        const int pc = (4 * half + c) ^ (row & 7);
        *reinterpret_cast<uint4 *>(base + pc * 16) = make_uint4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    }
}

}  // namespace gg
