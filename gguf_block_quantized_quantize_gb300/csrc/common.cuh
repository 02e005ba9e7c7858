// Device helpers shared by the CUDA kernels of libgguf_gb300 (sm_103a only).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gguf_gb300.h"

namespace gg {

// block geometry (public GGUF convention)
constexpr int QK8 = 32;            // values per Q8_0 / q8_1 block
constexpr int QKK = 256;           // values per K-quant super-block
constexpr int Q8_0_BYTES = 34;     // fp16 d, int8 q[32]
constexpr int Q8_1_BYTES = 36;     // fp16 d, fp16 s, int8 q[32]
constexpr int Q4_K_BYTES = 144;    // fp16 d, fp16 dmin, scales[12], qs[128]
constexpr int Q6_K_BYTES = 210;    // ql[128], qh[64], scales[16], fp16 d
constexpr int Q4_0_BYTES = 18;     // fp16 d, qs[16] (value l low nibble, l + 16 high)
constexpr int Q5_K_BYTES = 176;    // fp16 d, fp16 dmin, scales[12], qh[32], qs[128]
constexpr int MXFP4_BYTES = 17;    // u8 E8M0 exponent, qs[16] e2m1 codes (Q4_0's nibble order)

__device__ __forceinline__ float h2f(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ float bf2f(uint16_t h) { return __uint_as_float(((uint32_t)h) << 16); }

__device__ __forceinline__ uint16_t f2h_rn(float f) { return __half_as_ushort(__float2half_rn(f)); }
__device__ __forceinline__ uint16_t f2bf_rn(float f) { return __bfloat16_as_ushort(__float2bfloat16_rn(f)); }

// store one fp32 value as F32 / BF16 / F16 (round to nearest even)
__device__ __forceinline__ void store_out(void *out, int ot, int64_t idx, float v) {
    if (ot == GGUF_F32) reinterpret_cast<float *>(out)[idx] = v;
    else if (ot == GGUF_BF16) reinterpret_cast<uint16_t *>(out)[idx] = f2bf_rn(v);
    else reinterpret_cast<uint16_t *>(out)[idx] = f2h_rn(v);
}

// signed x signed 4-way byte dot product with accumulate
// Exact fp32 value of an integer on the full-rate pipes instead of the
// conversion unit (a quarter of the FMA rate or less): the bits of
// 1.5 * 2^23 + v are that float exactly while |v| < 2^22 (every per-block
// dot sum here: at most 32 * 255 * 127 in magnitude), and so are those of
// 2^23 + b for a byte b.
constexpr float kI2fBias = 12582912.0f;   // 1.5 * 2^23
__device__ __forceinline__ float i2f_bits(int v) { return __int_as_float(0x4B400000 + v); }   // = kI2fBias + v
__device__ __forceinline__ float i2f22(int v) { return i2f_bits(v) - kI2fBias; }
// byte i of w as an exact float
__device__ __forceinline__ float u8f(uint32_t w, int i) {
    return __uint_as_float(__byte_perm(w, 0x4B000000u, (uint32_t)i | (4u << 4) | (4u << 8) | (7u << 12))) - 8388608.0f;
}

__device__ __forceinline__ int dp4a_ss(int a, int b, int c) { return __dp4a(a, b, c); }

// asynchronous 4-byte global -> shared copy (both 4-byte aligned); the thread's
// copies are complete after cp_async_wait_all
__device__ __forceinline__ void cp_async4(void *sdst, const void *gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(sdst)), "l"(gsrc)
                 : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// unsigned (a) x signed (b) 4-way byte dot product with accumulate
__device__ __forceinline__ int dp4a_us(uint32_t a, int b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ uint32_t ld_u32(const uint8_t *p) { return *reinterpret_cast<const uint32_t *>(p); }
__device__ __forceinline__ uint16_t ld_u16(const uint8_t *p) { return *reinterpret_cast<const uint16_t *>(p); }

// Read 8 bytes at a 2-byte-aligned address as two words, touching only bytes
// in [p - 2, p + 10): aligned words plus a funnel shift when p % 4 == 2.
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

__device__ __forceinline__ void ld8_a2(const uint8_t *p, uint32_t &lo, uint32_t &hi) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint8_t *base = reinterpret_cast<const uint8_t *>(a & ~uintptr_t(3));
    uint32_t w0 = ld_u32(base), w1 = ld_u32(base + 4);
    if (a & 2) {
        uint32_t w2 = ld_u32(base + 8);
        lo = __funnelshift_r(w0, w1, 16);
        hi = __funnelshift_r(w1, w2, 16);
    } else {
        lo = w0;
        hi = w1;
    }
}

// 6-bit (scale, min) of Q4_K sub-block j from the 12 scale bytes held in three
// little-endian words sc[0..2] (bytes 0..11).
__device__ __forceinline__ int sc_byte(const uint32_t sc[3], int i) { return (sc[i >> 2] >> (8 * (i & 3))) & 0xff; }
__device__ __forceinline__ void q4k_scale_min(const uint32_t sc[3], int j, int &s, int &m) {
    if (j < 4) {
        s = sc_byte(sc, j) & 63;
        m = sc_byte(sc, j + 4) & 63;
    } else {
        s = (sc_byte(sc, j + 4) & 15) | ((sc_byte(sc, j - 4) >> 6) << 4);
        m = (sc_byte(sc, j + 4) >> 4) | ((sc_byte(sc, j) >> 6) << 4);
    }
}

// ---------------------------------------------------------------- MXFP4 helpers
// An MXFP4 value is e2m1(code) * 2^(e - 127).  Kernels carry the integer quant
// k = 2 * e2m1(code) (-12..12, exact) and the block factor 2^(e - 128).

// 2^(e - 128) for an E8M0 code e (exact: 2^-128 and 2^-127 are fp32 subnormals)
__device__ __forceinline__ float e8m0_half(uint32_t e) {
    return e >= 2 ? __uint_as_float((e - 1) << 23) : __uint_as_float(0x00200000u << e);
}

// The four e2m1 codes in the nibbles of the low 16 bits of s -> four bytes
// 16 + k (4..28), byte n from nibble n.  PRMT in its default mode takes table
// byte (code & 7) for a selector nibble whose top bit is clear and, where it
// is set, the replicated sign bit of that byte (0: the table bytes are
// non-negative).  So p holds k for the codes with the sign bit clear and q
// (sign bits flipped) |k| for the others, never both in one byte, and
// 16 + p - q needs no carry between bytes.
__device__ __forceinline__ uint32_t mxfp4_biased4(uint32_t s) {
    constexpr uint32_t T0 = 0x03020100u, T1 = 0x0C080604u;   // |k| of codes 0..7: 0 1 2 3 4 6 8 12
    const uint32_t s16 = s & 0xffffu;
    uint32_t p, q;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(p) : "r"(T0), "r"(T1), "r"(s16));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(q) : "r"(T0), "r"(T1), "r"(s16 ^ 0x8888u));
    return p + 0x10101010u - q;
}

// The 17 bytes of an MXFP4 block at any address p: the exponent byte e and the
// 16 code bytes as four words.  Reads only [p - 3, p + 17): four aligned words
// from p rounded down to 4, then single bytes up to p + 16.
__device__ __forceinline__ void ld_mxfp4_block(const uint8_t *p, uint32_t &e, uint32_t (&q)[4]) {
    const int off = (int)(reinterpret_cast<uintptr_t>(p) & 3);
    const uint8_t *b = p - off;
    uint32_t w[5];
#pragma unroll
    for (int i = 0; i < 4; i++) w[i] = ld_u32(b + 4 * i);
    uint32_t t = 0;
#pragma unroll
    for (int i = 0; i < 4; i++)
        if (i <= off) t |= (uint32_t)b[16 + i] << (8 * i);
    w[4] = t;
    e = (w[0] >> (8 * off)) & 0xffu;
    const int s = off + 1;   // the code bytes start at b + s
#pragma unroll
    for (int j = 0; j < 4; j++) q[j] = s == 4 ? w[j + 1] : __funnelshift_r(w[j], w[j + 1], 8 * s);
}

// k = 2 * e2m1(code) for one code, by its fields (sign, exponent, mantissa)
__device__ __forceinline__ int mxfp4_k(uint32_t c) {
    const int c7 = (int)(c & 7);
    const int mag = c7 < 4 ? c7 : (2 + (c7 & 1)) << ((c7 >> 1) - 1);
    return (c & 8) ? -mag : mag;
}

__host__ __device__ constexpr int64_t block_elems(int t) {
    return (t == GGUF_Q8_0 || t == GGUF_Q8_1 || t == GGUF_Q4_0 || t == GGUF_MXFP4) ? 32
         : (t == GGUF_Q4_K || t == GGUF_Q5_K || t == GGUF_Q6_K) ? 256
         : (t == GGUF_F32 || t == GGUF_F16 || t == GGUF_BF16) ? 1 : 0;
}
__host__ __device__ constexpr int64_t block_bytes(int t) {
    return t == GGUF_Q8_0 ? 34 : t == GGUF_Q8_1 ? 36 : t == GGUF_Q4_K ? 144 : t == GGUF_Q6_K ? 210
         : t == GGUF_Q4_0 ? 18 : t == GGUF_Q5_K ? 176 : t == GGUF_MXFP4 ? 17
         : t == GGUF_F32 ? 4 : (t == GGUF_F16 || t == GGUF_BF16) ? 2 : 0;
}

}  // namespace gg
