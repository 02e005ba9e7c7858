/*
 * gguf_oracle.c -- plain, slow, scalar CPU oracle for the GGUF block-quantized
 * matmul path (q8_1 activations x Q8_0 / Q4_0 / Q4_1 / Q5_0 / Q5_1 / Q4_K /
 * Q5_K / Q6_K / MXFP4 weights).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or runs
 * this file: only tests/, __graft_entry__.smoke() and the cpu_baseline leg of
 * bench.py may.  It shares no source, header, table or helper with the CUDA
 * library; it is compiled on its own with -ffp-contract=off so that every fp32
 * operation below is one IEEE operation, in the order written.
 *
 * What it computes, and where the pages say so:
 *  - Activations (fp32 / bf16 / fp16) are quantized "to q8_1 directly" and the
 *    result is accumulated in fp32 and returned in the activation dtype
 *    (FreeToken PR #690 "serve GGUF checkpoints on vendored ggml-cuda kernels",
 *    section "Vendored ggml", list "What the ggml patch changes").
 *  - K-quant super-blocks span K = 256 (1Cat-vLLM "GGUF on V100: implementation
 *    and acceptance control", section "TP/EP decision"); Q4_K is affine, a scale
 *    plus an additive min (same page, "Repack admission finding: Q4_K affine
 *    coefficients").
 *  - mul_mat_id, fused GLU, MoE weighted sum, get_rows and dequantize are the op
 *    list of FreeToken PR #690 (section "Vendored ggml", paragraph "Our own code
 *    next to it"); repeated expert ids within a token and inactive slots must
 *    be handled (FreeToken issue #671 "MoE cache, CPU experts and GGUF support",
 *    section "Known issues").
 *
 * Readings where the pages are silent (the pages name the formats but never
 * print their bytes):
 *  - MXFP4 is another type the pages list (FreeToken PR #690, "Tensor types").
 *    Its values are OCP microscaling FP4: e2m1 codes (sign, 2-bit exponent,
 *    1-bit mantissa) scaled by the block's E8M0 exponent, 2^(e - 127); the
 *    GGUF block is {u8 e, u8 qs[16]} with Q4_0's nibble order.  E8M0 code 255
 *    (NaN in the OCP definition) is read as the exponent 128 like any other.
 *  - Q4_1, Q5_0 and Q5_1 are listed there too.  Their public GGUF blocks of 32:
 *    Q4_1 {fp16 d, fp16 m, qs[16]}, value d*q + m; Q5_0 {fp16 d, qh[4],
 *    qs[16]}, value d*(q - 16); Q5_1 {fp16 d, fp16 m, qh[4], qs[16]}, value
 *    d*q + m.  The nibbles are in Q4_0's order; the fifth bit of value i is
 *    bit i of qh read as a little-endian 32-bit word.
 *  - Q4_0 and Q5_K are two of the further tensor types the pages list
 *    (FreeToken PR #690, "Tensor types"; transformers PR #45977, supported
 *    quant types of GgufLinear).
 *  - Byte layouts of Q8_0 / q8_1 / Q4_0 / Q4_K / Q5_K / Q6_K follow the public GGUF
 *    convention, so that blocks stay GGUF-compatible.  Layout parity with real
 *    GGUF files is unpinned (no GGUF file or gguf-py exists here); everything
 *    else is pinned by the tests in tests/test_oracle_*.py.
 *  - q8_1: d = amax / 127 (one IEEE fp32 division), q = roundf(x / d) (half
 *    away from zero), s = fp16(d * (float)sum(q)) with the fp32 d.
 *  - dequantized value order: Q4_K, Q5_K  a = d*s; b = dmin*m; v = a*q - b;
 *                             Q6_K  v = (d*sc) * (q - 32);   Q8_0  v = d*q;
 *                             Q4_0  v = d * (q - 8);   Q5_0  v = d * (q - 16);
 *                             Q4_1, Q5_1  v = d*q + m (one rounding);
 *                             MXFP4 v = e2m1(q) * 2^(e - 127), one exact product.
 *  - block dots: symmetric formats with an integer offset (Q4_0: 8, Q5_0: 16,
 *    Q6_K: 32) take the offset into the exact integer sum; affine formats with
 *    a float min (Q4_K, Q5_K: -dmin*m_j; Q4_1, Q5_1: +m) combine the min with
 *    the activation block's stored s.
 *    MXFP4's integer quant is 2 * e2m1(q) (exact, in -12..12) against the
 *    block factor 2^(e - 128).
 *  - matmul reference: the blockwise formula evaluated in fp64 on the stored
 *    (fp16) fields, e.g. Q4_K y = sum_j (d*s_j*d_a*S_j - dmin*m_j*s_a).
 *  - weight quantizers (test-input generators only; the GPU never quantizes
 *    weights) are the simple deterministic ones described at each function.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include "gguf_oracle.h"

/* ------------------------------------------------------------------------ */
/* IEEE binary16 / bfloat16 <-> binary32, written from the format definitions */
/* ------------------------------------------------------------------------ */

float orc_f16_to_f32(uint16_t h) {
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 31;
    int man = h & 1023;
    float v;
    if (exp == 0) {
        v = ldexpf((float)man, -24); /* subnormal: man * 2^-24 */
    } else if (exp == 31) {
        v = man ? NAN : INFINITY;
    } else {
        v = ldexpf((float)(man + 1024), exp - 25); /* (1024+man) * 2^(exp-15-10) */
    }
    return sign ? -v : v;
}

/* Round-to-nearest-even of a non-negative double q that is an exact multiple
 * of 2^-30 or coarser (always true here: q is a float scaled by a power of 2). */
static double orc_rne(double q) {
    double fl = floor(q);
    double diff = q - fl;
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

uint16_t orc_f32_to_f16(float f) {
    if (isnan(f)) return 0x7e00;
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs((double)f);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    e -= 1;             /* a = (2m) * 2^e, 2m in [1, 2) */
    if (e < -14) e = -14; /* below the normal range the quantum stays 2^-24 */
    if (e > 15) return sign | 0x7c00;
    double quantum = ldexp(1.0, e - 10);
    double r = orc_rne(a / quantum); /* exact division by a power of two */
    if (r >= 2048.0) { r = 1024.0; e += 1; }
    if (e > 15) return sign | 0x7c00;
    if (r < 1024.0) return sign | (uint16_t)r; /* subnormal (e == -14) */
    return sign | (uint16_t)(((e + 15) << 10) | ((int)r - 1024));
}

float orc_bf16_to_f32(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* round-to-nearest-even of an fp64 value to bf16, in one step (no fp32 hop) */
uint16_t orc_f64_to_bf16(double f) {
    if (isnan(f)) return 0x7fc0;
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs(f);
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);
    e -= 1;
    if (e < -126) e = -126; /* bf16 shares fp32's exponent range */
    double quantum = ldexp(1.0, e - 7);
    double r = orc_rne(a / quantum);
    if (r >= 256.0) { r = 128.0; e += 1; }
    if (e > 127) return sign | 0x7f80;
    if (r < 128.0) return sign | (uint16_t)r; /* subnormal */
    return sign | (uint16_t)(((e + 127) << 7) | ((int)r - 128));
}

/* every fp32 value is an fp64 value: the same rounding */
uint16_t orc_f32_to_bf16(float f) { return orc_f64_to_bf16((double)f); }

static uint16_t rd16(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t *p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }

/* ------------------------------------------------------------------------ */
/* type table                                                               */
/* ------------------------------------------------------------------------ */

int64_t orc_block_elems(int type) {
    switch (type) {
    case ORC_F32: case ORC_F16: case ORC_BF16: return 1;
    case ORC_Q8_0: case ORC_Q8_1: case ORC_Q4_0: case ORC_MXFP4:
    case ORC_Q4_1: case ORC_Q5_0: case ORC_Q5_1: return 32;
    case ORC_Q4_K: case ORC_Q5_K: case ORC_Q6_K: return 256;
    default: return 0;
    }
}

int64_t orc_block_bytes(int type) {
    switch (type) {
    case ORC_F32: return 4;
    case ORC_F16: case ORC_BF16: return 2;
    case ORC_Q8_0: return 34;  /* fp16 d, int8 q[32] */
    case ORC_Q8_1: return 36;  /* fp16 d, fp16 s, int8 q[32] */
    case ORC_Q4_0: return 18;  /* fp16 d, u8 qs[16] */
    case ORC_MXFP4: return 17; /* u8 e (E8M0), u8 qs[16] (e2m1 codes) */
    case ORC_Q4_1: return 20;  /* fp16 d, fp16 m, u8 qs[16] */
    case ORC_Q5_0: return 22;  /* fp16 d, u8 qh[4], u8 qs[16] */
    case ORC_Q5_1: return 24;  /* fp16 d, fp16 m, u8 qh[4], u8 qs[16] */
    case ORC_Q4_K: return 144; /* fp16 d, fp16 dmin, u8 scales[12], u8 qs[128] */
    case ORC_Q5_K: return 176; /* fp16 d, fp16 dmin, u8 scales[12], u8 qh[32], u8 qs[128] */
    case ORC_Q6_K: return 210; /* u8 ql[128], u8 qh[64], i8 scales[16], fp16 d */
    default: return 0;
    }
}

int64_t orc_row_size(int type, int64_t k) {
    int64_t be = orc_block_elems(type);
    if (be == 0 || k % be) return -1;
    return k / be * orc_block_bytes(type);
}

/* sub-block length of the per-block integer dot products */
int64_t orc_sub_elems(int type) {
    switch (type) {
    case ORC_Q8_0: case ORC_Q4_0: case ORC_Q4_K: case ORC_Q5_K: case ORC_MXFP4:
    case ORC_Q4_1: case ORC_Q5_0: case ORC_Q5_1: return 32;
    case ORC_Q6_K: return 16;
    default: return 0;
    }
}

/* ------------------------------------------------------------------------ */
/* field accessors: the only place that knows the bytes of each format      */
/* ------------------------------------------------------------------------ */

/* Q8_0 block: value i = d * q[i] */
static float q8_0_d(const uint8_t *b) { return orc_f16_to_f32(rd16(b)); }
static int q8_0_q(const uint8_t *b, int i) { return (int8_t)b[2 + i]; }

/* q8_1 block: value i = d * q[i]; s is the stored fp16 of d * sum(q) */
static float q8_1_d(const uint8_t *b) { return orc_f16_to_f32(rd16(b)); }
static float q8_1_s(const uint8_t *b) { return orc_f16_to_f32(rd16(b + 2)); }
static int q8_1_q(const uint8_t *b, int i) { return (int8_t)b[4 + i]; }

/* Q4_K super-block.  The 6-bit (scale, min) of sub-block j (0..7):
 *   j < 4 : scale = sc[j] & 63,                  min = sc[j+4] & 63
 *   j >= 4: scale = (sc[j+4] & 15) | (sc[j-4] >> 6) << 4,
 *           min   = (sc[j+4] >> 4) | (sc[j]   >> 6) << 4                     */
static float q4_k_d(const uint8_t *b) { return orc_f16_to_f32(rd16(b)); }
static float q4_k_dmin(const uint8_t *b) { return orc_f16_to_f32(rd16(b + 2)); }
static void q4_k_scale_min(const uint8_t *b, int j, int *s, int *m) {
    const uint8_t *sc = b + 4;
    if (j < 4) {
        *s = sc[j] & 63;
        *m = sc[j + 4] & 63;
    } else {
        *s = (sc[j + 4] & 15) | ((sc[j - 4] >> 6) << 4);
        *m = (sc[j + 4] >> 4) | ((sc[j] >> 6) << 4);
    }
}
/* value i (0..255): chunk c = i / 64 uses qs[32c .. 32c+31]; the low nibble of
 * qs[32c + l] is value 64c + l, the high nibble is value 64c + 32 + l.       */
static int q4_k_q(const uint8_t *b, int i) {
    const uint8_t *qs = b + 16;
    int c = i / 64, r = i % 64;
    uint8_t byte = qs[32 * c + (r % 32)];
    return r < 32 ? (byte & 15) : (byte >> 4);
}

/* Q4_0 block: 32 unsigned 4-bit quants; byte qs[l] (l = 0..15) holds value l
 * in its low nibble and value l + 16 in its high nibble; value = d * (q - 8). */
static float q4_0_d(const uint8_t *b) { return orc_f16_to_f32(rd16(b)); }
static int q4_0_q(const uint8_t *b, int i) {
    uint8_t byte = b[2 + (i % 16)];
    return i < 16 ? (byte & 15) : (byte >> 4);
}

/* Q4_1 / Q5_0 / Q5_1 blocks of 32.  The quant bytes qs (16) hold value l in
 * the low nibble of qs[l] and value l + 16 in the high one; Q5_0 / Q5_1 add
 * bit i of the little-endian word qh as bit 4 of value i.                    */
static int qs_nibble(const uint8_t *qs, int i) { return i < 16 ? (qs[i] & 15) : (qs[i - 16] >> 4); }
static int qh_bit(const uint8_t *qh, int i) { return (qh[i / 8] >> (i % 8)) & 1; }
static float q41_d(const uint8_t *b) { return orc_f16_to_f32(rd16(b)); }
static float q41_m(const uint8_t *b) { return orc_f16_to_f32(rd16(b + 2)); }
static int q4_1_q(const uint8_t *b, int i) { return qs_nibble(b + 4, i); }
static float q5_0_d(const uint8_t *b) { return orc_f16_to_f32(rd16(b)); }
static int q5_0_q(const uint8_t *b, int i) { return qs_nibble(b + 6, i) | (qh_bit(b + 2, i) << 4); }
static int q5_1_q(const uint8_t *b, int i) { return qs_nibble(b + 8, i) | (qh_bit(b + 4, i) << 4); }

/* MXFP4 block: byte 0 is the E8M0 exponent e, bytes 1..16 hold 32 e2m1 codes
 * in Q4_0's order (byte 1 + l: code of value l low, of value l + 16 high).
 * e2m1 code c: sign c >> 3, exponent E = (c >> 1) & 3, mantissa M = c & 1;
 * magnitude M / 2 when E = 0 (subnormal), else 2^(E - 1) * (1 + M / 2).     */
static int mxfp4_e(const uint8_t *b) { return b[0]; }
static int mxfp4_code(const uint8_t *b, int i) {
    uint8_t byte = b[1 + (i % 16)];
    return i < 16 ? (byte & 15) : (byte >> 4);
}
static double e2m1_value(int c) {
    int E = (c >> 1) & 3, M = c & 1;
    double mag = E == 0 ? 0.5 * M : ldexp(1.0 + 0.5 * M, E - 1);
    return (c & 8) ? -mag : mag;
}
/* the integer quant 2 * e2m1(c), exact in -12..12 */
static int mxfp4_q(const uint8_t *b, int i) { return (int)(2.0 * e2m1_value(mxfp4_code(b, i))); }

/* Q5_K super-block: the header (d, dmin, 12 scale bytes) is packed exactly as
 * Q4_K's, so q4_k_d / q4_k_dmin / q4_k_scale_min read it too.  Value i takes
 * its low 4 bits from qs (at byte 48) as Q4_K takes its quant from qs at 16,
 * and its fifth bit from qh[i % 32] (at byte 16), bit i / 32 -- the sub-block
 * index.  q in 0..31; value = d*s_j*q - dmin*m_j.                           */
static int q5_k_q(const uint8_t *b, int i) {
    const uint8_t *qs = b + 48, *qh = b + 16;
    int c = i / 64, r = i % 64;
    uint8_t byte = qs[32 * c + (r % 32)];
    int lo = r < 32 ? (byte & 15) : (byte >> 4);
    int hi = (qh[i % 32] >> (i / 32)) & 1;
    return lo | (hi << 4);
}

/* Q6_K super-block.  Half h = i / 128 uses ql + 64h, qh + 32h, sc + 8h.  For
 * o = i % 128, l = o % 32, g = o / 32: the low 4 bits come from
 *   g=0: ql[l] & 15   g=1: ql[l+32] & 15   g=2: ql[l] >> 4   g=3: ql[l+32] >> 4
 * and the high 2 bits are bits (2g, 2g+1) of qh[l].  q in 0..63;
 * value = d * sc[8h + o/16] * (q - 32).                                      */
static float q6_k_d(const uint8_t *b) { return orc_f16_to_f32(rd16(b + 208)); }
static int q6_k_scale(const uint8_t *b, int i) {
    int h = i / 128, o = i % 128;
    return (int8_t)b[192 + 8 * h + o / 16];
}
static int q6_k_q(const uint8_t *b, int i) {
    int h = i / 128, o = i % 128, l = o % 32, g = o / 32;
    const uint8_t *ql = b + 64 * h;
    const uint8_t *qh = b + 128 + 32 * h;
    int lo = (g == 0) ? (ql[l] & 15) : (g == 1) ? (ql[l + 32] & 15) : (g == 2) ? (ql[l] >> 4) : (ql[l + 32] >> 4);
    int hi = (qh[l] >> (2 * g)) & 3;
    return lo | (hi << 4);
}

/* ------------------------------------------------------------------------ */
/* activation quantizer: fp32 -> q8_1                                        */
/* ------------------------------------------------------------------------ */

void orc_quantize_q8_1_block(const float *x, uint8_t *out) {
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    int sum = 0;
    for (int i = 0; i < 32; i++) {
        int q = 0;
        if (d != 0.0f) q = (int)roundf(x[i] / d);
        out[4 + i] = (uint8_t)(int8_t)q;
        sum += q;
    }
    float s = d * (float)sum;
    wr16(out, orc_f32_to_f16(d));
    wr16(out + 2, orc_f32_to_f16(s));
}

/* x: m rows of k fp32 values (row stride ldx elements) -> m rows of k/32 q8_1 blocks */
int orc_quantize_q8_1(const float *x, int64_t m, int64_t k, int64_t ldx, uint8_t *out) {
    if (k % 32) return -1;
    int64_t rb = k / 32 * 36;
    for (int64_t r = 0; r < m; r++)
        for (int64_t b = 0; b < k / 32; b++)
            orc_quantize_q8_1_block(x + r * ldx + b * 32, out + r * rb + b * 36);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* weight quantizers (test-input generation only)                           */
/* ------------------------------------------------------------------------ */

/* Q8_0: d = amax / 127, q = clamp(roundf(x / d), -127, 127) with the fp32 d. */
static void quantize_block_q8_0(const float *x, uint8_t *out) {
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    for (int i = 0; i < 32; i++) {
        int q = 0;
        if (d != 0.0f) q = (int)roundf(x[i] / d);
        if (q > 127) q = 127;
        if (q < -127) q = -127;
        out[2 + i] = (uint8_t)(int8_t)q;
    }
    wr16(out, orc_f32_to_f16(d));
}

/* Q4_K: per sub-block j of 32, lo = min(0, min x), hi = max x,
 * scale_j = (hi - lo) / 15, min_j = -lo; d = max scale / 63, dmin = max min / 63;
 * 6-bit s_j = roundf(scale_j / d), m_j = roundf(min_j / dmin);
 * q = clamp(roundf((x + dmin_h * m_j) / (d_h * s_j)), 0, 15) with the stored
 * (fp16) d_h, dmin_h.  Scale-search refinements of other quantizers change only
 * the quality of the test weights, not the format.                          */
static void quantize_block_q4_k(const float *x, uint8_t *out) {
    float scale[8], minv[8];
    float maxscale = 0.0f, maxmin = 0.0f;
    for (int j = 0; j < 8; j++) {
        float lo = 0.0f, hi = x[32 * j];
        for (int i = 0; i < 32; i++) {
            float v = x[32 * j + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        scale[j] = (hi - lo) / 15.0f;
        minv[j] = -lo;
        if (scale[j] > maxscale) maxscale = scale[j];
        if (minv[j] > maxmin) maxmin = minv[j];
    }
    float d = maxscale / 63.0f, dmin = maxmin / 63.0f;
    int s6[8], m6[8];
    for (int j = 0; j < 8; j++) {
        int s = d > 0.0f ? (int)roundf(scale[j] / d) : 0;
        int m = dmin > 0.0f ? (int)roundf(minv[j] / dmin) : 0;
        s6[j] = s > 63 ? 63 : s;
        m6[j] = m > 63 ? 63 : m;
    }
    uint16_t dh = orc_f32_to_f16(d), dminh = orc_f32_to_f16(dmin);
    float df = orc_f16_to_f32(dh), dminf = orc_f16_to_f32(dminh);
    memset(out, 0, 144);
    wr16(out, dh);
    wr16(out + 2, dminh);
    uint8_t *sc = out + 4;
    for (int j = 0; j < 8; j++) {
        if (j < 4) {
            sc[j] |= (uint8_t)s6[j];
            sc[j + 4] |= (uint8_t)m6[j];
        } else {
            sc[j + 4] |= (uint8_t)((s6[j] & 15) | ((m6[j] & 15) << 4));
            sc[j - 4] |= (uint8_t)((s6[j] >> 4) << 6);
            sc[j] |= (uint8_t)((m6[j] >> 4) << 6);
        }
    }
    uint8_t *qs = out + 16;
    for (int i = 0; i < 256; i++) {
        int j = i / 32;
        float denom = df * (float)s6[j];
        int q = 0;
        if (denom > 0.0f) q = (int)roundf((x[i] + dminf * (float)m6[j]) / denom);
        if (q < 0) q = 0;
        if (q > 15) q = 15;
        int c = i / 64, r = i % 64;
        if (r < 32) qs[32 * c + r] |= (uint8_t)q;
        else qs[32 * c + r - 32] |= (uint8_t)(q << 4);
    }
}

/* Q4_0: the value v of largest magnitude sets d = v / -8 (so that v maps to
 * q - 8 = -8); q = clamp(roundf(x / d) + 8, 0, 15) with the stored (fp16) d. */
static void quantize_block_q4_0(const float *x, uint8_t *out) {
    float amax = 0.0f, vmax = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(x[i]);
        if (a > amax) { amax = a; vmax = x[i]; }
    }
    uint16_t dh = orc_f32_to_f16(vmax / -8.0f);
    float df = orc_f16_to_f32(dh);
    memset(out, 0, 18);
    wr16(out, dh);
    for (int i = 0; i < 32; i++) {
        int q = 8;
        if (df != 0.0f) q = (int)roundf(x[i] / df) + 8;
        if (q < 0) q = 0;
        if (q > 15) q = 15;
        out[2 + (i % 16)] |= (uint8_t)(i < 16 ? q : q << 4);
    }
}

/* Q4_1 / Q5_1 (levels = 15 / 31): m = min x, d = (max x - m) / levels; the
 * stored fp16 d_h, m_h; q = clamp(roundf((x - m_h) / d_h), 0, levels).
 * Q5_0: the value v of largest magnitude sets d = v / -16;
 * q = clamp(roundf(x / d_h) + 16, 0, 31).                                   */
static void quantize_block_affine32(const float *x, uint8_t *out, int levels, int with_qh) {
    float lo = x[0], hi = x[0];
    for (int i = 1; i < 32; i++) {
        if (x[i] < lo) lo = x[i];
        if (x[i] > hi) hi = x[i];
    }
    uint16_t dh = orc_f32_to_f16((hi - lo) / (float)levels), mh = orc_f32_to_f16(lo);
    float df = orc_f16_to_f32(dh), mf = orc_f16_to_f32(mh);
    int bytes = with_qh ? 24 : 20;
    memset(out, 0, (size_t)bytes);
    wr16(out, dh);
    wr16(out + 2, mh);
    uint8_t *qh = out + 4, *qs = out + (with_qh ? 8 : 4);
    for (int i = 0; i < 32; i++) {
        int q = 0;
        if (df > 0.0f) q = (int)roundf((x[i] - mf) / df);
        if (q < 0) q = 0;
        if (q > levels) q = levels;
        qs[i % 16] |= (uint8_t)(i < 16 ? (q & 15) : (q & 15) << 4);
        if (with_qh) qh[i / 8] |= (uint8_t)(((q >> 4) & 1) << (i % 8));
    }
}
static void quantize_block_q5_0(const float *x, uint8_t *out) {
    float amax = 0.0f, vmax = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(x[i]);
        if (a > amax) { amax = a; vmax = x[i]; }
    }
    uint16_t dh = orc_f32_to_f16(vmax / -16.0f);
    float df = orc_f16_to_f32(dh);
    memset(out, 0, 22);
    wr16(out, dh);
    for (int i = 0; i < 32; i++) {
        int q = 16;
        if (df != 0.0f) q = (int)roundf(x[i] / df) + 16;
        if (q < 0) q = 0;
        if (q > 31) q = 31;
        out[6 + (i % 16)] |= (uint8_t)(i < 16 ? (q & 15) : (q & 15) << 4);
        out[2 + i / 8] |= (uint8_t)(((q >> 4) & 1) << (i % 8));
    }
}

/* MXFP4: the smallest e in 0..254 with 6 * 2^(e - 127) >= amax (0 for an
 * all-zero block), then per value the e2m1 code of the nearest magnitude of
 * |x| / 2^(e - 127) (ties to the larger), with x's sign.                     */
static void quantize_block_mxfp4(const float *x, uint8_t *out) {
    double amax = 0.0;
    for (int i = 0; i < 32; i++) {
        double a = fabs((double)x[i]);
        if (a > amax) amax = a;
    }
    int e = 0;
    while (e < 254 && 6.0 * ldexp(1.0, e - 127) < amax) e++;
    memset(out, 0, 17);
    out[0] = (uint8_t)e;
    double s = ldexp(1.0, e - 127);
    for (int i = 0; i < 32; i++) {
        double r = fabs((double)x[i]) / s;
        int best = 0;
        for (int c = 1; c < 8; c++) {
            double dc = fabs(e2m1_value(c) - r), db = fabs(e2m1_value(best) - r);
            if (dc <= db) best = c;
        }
        if (x[i] < 0.0f && best != 0) best |= 8;
        out[1 + (i % 16)] |= (uint8_t)(i < 16 ? best : best << 4);
    }
}

/* Q5_K: as Q4_K with 32 levels: scale_j = (hi - lo) / 31, q in 0..31, the low
 * 4 bits packed as Q4_K's quants (at byte 48) and bit 4 of value i set as bit
 * i / 32 of qh[i % 32].                                                      */
static void quantize_block_q5_k(const float *x, uint8_t *out) {
    float scale[8], minv[8];
    float maxscale = 0.0f, maxmin = 0.0f;
    for (int j = 0; j < 8; j++) {
        float lo = 0.0f, hi = x[32 * j];
        for (int i = 0; i < 32; i++) {
            float v = x[32 * j + i];
            if (v < lo) lo = v;
            if (v > hi) hi = v;
        }
        scale[j] = (hi - lo) / 31.0f;
        minv[j] = -lo;
        if (scale[j] > maxscale) maxscale = scale[j];
        if (minv[j] > maxmin) maxmin = minv[j];
    }
    float d = maxscale / 63.0f, dmin = maxmin / 63.0f;
    int s6[8], m6[8];
    for (int j = 0; j < 8; j++) {
        int s = d > 0.0f ? (int)roundf(scale[j] / d) : 0;
        int m = dmin > 0.0f ? (int)roundf(minv[j] / dmin) : 0;
        s6[j] = s > 63 ? 63 : s;
        m6[j] = m > 63 ? 63 : m;
    }
    uint16_t dh = orc_f32_to_f16(d), dminh = orc_f32_to_f16(dmin);
    float df = orc_f16_to_f32(dh), dminf = orc_f16_to_f32(dminh);
    memset(out, 0, 176);
    wr16(out, dh);
    wr16(out + 2, dminh);
    uint8_t *sc = out + 4;
    for (int j = 0; j < 8; j++) {
        if (j < 4) {
            sc[j] |= (uint8_t)s6[j];
            sc[j + 4] |= (uint8_t)m6[j];
        } else {
            sc[j + 4] |= (uint8_t)((s6[j] & 15) | ((m6[j] & 15) << 4));
            sc[j - 4] |= (uint8_t)((s6[j] >> 4) << 6);
            sc[j] |= (uint8_t)((m6[j] >> 4) << 6);
        }
    }
    uint8_t *qh = out + 16, *qs = out + 48;
    for (int i = 0; i < 256; i++) {
        int j = i / 32;
        float denom = df * (float)s6[j];
        int q = 0;
        if (denom > 0.0f) q = (int)roundf((x[i] + dminf * (float)m6[j]) / denom);
        if (q < 0) q = 0;
        if (q > 31) q = 31;
        int c = i / 64, r = i % 64;
        if (r < 32) qs[32 * c + r] |= (uint8_t)(q & 15);
        else qs[32 * c + r - 32] |= (uint8_t)((q & 15) << 4);
        qh[i % 32] |= (uint8_t)((q >> 4) << (i / 32));
    }
}

/* Q6_K: per sub-block j of 16, scale_j = amax_j / 31; d = max scale / 127;
 * sc_j = roundf(scale_j / d); q = clamp(roundf(x / (d_h * sc_j)), -32, 31) + 32. */
static void quantize_block_q6_k(const float *x, uint8_t *out) {
    float scale[16], maxs = 0.0f;
    for (int j = 0; j < 16; j++) {
        float amax = 0.0f;
        for (int i = 0; i < 16; i++) {
            float a = fabsf(x[16 * j + i]);
            if (a > amax) amax = a;
        }
        scale[j] = amax / 31.0f;
        if (scale[j] > maxs) maxs = scale[j];
    }
    float d = maxs / 127.0f;
    int sc[16];
    for (int j = 0; j < 16; j++) {
        int s = d > 0.0f ? (int)roundf(scale[j] / d) : 0;
        sc[j] = s > 127 ? 127 : s;
    }
    uint16_t dh = orc_f32_to_f16(d);
    float df = orc_f16_to_f32(dh);
    memset(out, 0, 210);
    for (int j = 0; j < 16; j++) out[192 + j] = (uint8_t)(int8_t)sc[j];
    wr16(out + 208, dh);
    for (int i = 0; i < 256; i++) {
        float denom = df * (float)sc[i / 16];
        int q = 0;
        if (denom != 0.0f) q = (int)roundf(x[i] / denom);
        if (q < -32) q = -32;
        if (q > 31) q = 31;
        q += 32;
        int h = i / 128, o = i % 128, l = o % 32, g = o / 32;
        uint8_t *ql = out + 64 * h;
        uint8_t *qh = out + 128 + 32 * h;
        int lo = q & 15, hi = q >> 4;
        if (g == 0) ql[l] |= (uint8_t)lo;
        else if (g == 1) ql[l + 32] |= (uint8_t)lo;
        else if (g == 2) ql[l] |= (uint8_t)(lo << 4);
        else ql[l + 32] |= (uint8_t)(lo << 4);
        qh[l] |= (uint8_t)(hi << (2 * g));
    }
}

/* w: n rows of k fp32 values -> n packed rows of the given weight type */
int orc_quantize_weights(int type, const float *w, int64_t n, int64_t k, uint8_t *out) {
    int64_t rs = orc_row_size(type, k);
    if (rs < 0) return -1;
    int64_t be = orc_block_elems(type), bb = orc_block_bytes(type);
    for (int64_t r = 0; r < n; r++) {
        for (int64_t b = 0; b < k / be; b++) {
            const float *x = w + r * k + b * be;
            uint8_t *o = out + r * rs + b * bb;
            switch (type) {
            case ORC_Q8_0: quantize_block_q8_0(x, o); break;
            case ORC_Q4_0: quantize_block_q4_0(x, o); break;
            case ORC_MXFP4: quantize_block_mxfp4(x, o); break;
            case ORC_Q4_1: quantize_block_affine32(x, o, 15, 0); break;
            case ORC_Q5_1: quantize_block_affine32(x, o, 31, 1); break;
            case ORC_Q5_0: quantize_block_q5_0(x, o); break;
            case ORC_Q4_K: quantize_block_q4_k(x, o); break;
            case ORC_Q5_K: quantize_block_q5_k(x, o); break;
            case ORC_Q6_K: quantize_block_q6_k(x, o); break;
            case ORC_Q8_1: orc_quantize_q8_1_block(x, o); break;
            default: return -1;
            }
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* dequantization (fp32, fixed operation order)                             */
/* ------------------------------------------------------------------------ */

static float dequant_value(int type, const uint8_t *blk, int i) {
    switch (type) {
    case ORC_Q8_0: return q8_0_d(blk) * (float)q8_0_q(blk, i);
    case ORC_Q8_1: return q8_1_d(blk) * (float)q8_1_q(blk, i);
    case ORC_Q4_K: {
        int s, m;
        q4_k_scale_min(blk, i / 32, &s, &m);
        float a = q4_k_d(blk) * (float)s;
        float b = q4_k_dmin(blk) * (float)m;
        return a * (float)q4_k_q(blk, i) - b;
    }
    case ORC_Q4_0: return q4_0_d(blk) * (float)(q4_0_q(blk, i) - 8);
    case ORC_MXFP4: return ldexpf((float)e2m1_value(mxfp4_code(blk, i)), mxfp4_e(blk) - 127);
    case ORC_Q4_1: return q41_d(blk) * (float)q4_1_q(blk, i) + q41_m(blk);
    case ORC_Q5_0: return q5_0_d(blk) * (float)(q5_0_q(blk, i) - 16);
    case ORC_Q5_1: return q41_d(blk) * (float)q5_1_q(blk, i) + q41_m(blk);
    case ORC_Q5_K: {
        int s, m;
        q4_k_scale_min(blk, i / 32, &s, &m);
        float a = q4_k_d(blk) * (float)s;
        float b = q4_k_dmin(blk) * (float)m;
        return a * (float)q5_k_q(blk, i) - b;
    }
    case ORC_Q6_K: {
        float a = q6_k_d(blk) * (float)q6_k_scale(blk, i);
        return a * (float)(q6_k_q(blk, i) - 32);
    }
    default: return NAN;
    }
}

int orc_dequantize_row(int type, const uint8_t *row, int64_t k, float *out) {
    int64_t be = orc_block_elems(type), bb = orc_block_bytes(type);
    if (be < 32 || k % be) return -1;
    for (int64_t b = 0; b < k / be; b++)
        for (int64_t i = 0; i < be; i++) out[b * be + i] = dequant_value(type, row + b * bb, (int)i);
    return 0;
}

/* Same values in fp64 (every factor is an exact fp32 value; no rounding).    */
static double dequant_value_f64(int type, const uint8_t *blk, int i) {
    switch (type) {
    case ORC_Q8_0: return (double)q8_0_d(blk) * (double)q8_0_q(blk, i);
    case ORC_Q8_1: return (double)q8_1_d(blk) * (double)q8_1_q(blk, i);
    case ORC_Q4_K: {
        int s, m;
        q4_k_scale_min(blk, i / 32, &s, &m);
        return (double)q4_k_d(blk) * s * q4_k_q(blk, i) - (double)q4_k_dmin(blk) * m;
    }
    case ORC_Q4_0: return (double)q4_0_d(blk) * (q4_0_q(blk, i) - 8);
    case ORC_MXFP4: return ldexp(e2m1_value(mxfp4_code(blk, i)), mxfp4_e(blk) - 127);
    case ORC_Q4_1: return (double)q41_d(blk) * q4_1_q(blk, i) + (double)q41_m(blk);
    case ORC_Q5_0: return (double)q5_0_d(blk) * (q5_0_q(blk, i) - 16);
    case ORC_Q5_1: return (double)q41_d(blk) * q5_1_q(blk, i) + (double)q41_m(blk);
    case ORC_Q5_K: {
        int s, m;
        q4_k_scale_min(blk, i / 32, &s, &m);
        return (double)q4_k_d(blk) * s * q5_k_q(blk, i) - (double)q4_k_dmin(blk) * m;
    }
    case ORC_Q6_K: return (double)q6_k_d(blk) * q6_k_scale(blk, i) * (q6_k_q(blk, i) - 32);
    default: return NAN;
    }
}

int orc_dequantize_row_f64(int type, const uint8_t *row, int64_t k, double *out) {
    int64_t be = orc_block_elems(type), bb = orc_block_bytes(type);
    if (be < 32 || k % be) return -1;
    for (int64_t b = 0; b < k / be; b++)
        for (int64_t i = 0; i < be; i++) out[b * be + i] = dequant_value_f64(type, row + b * bb, (int)i);
    return 0;
}

/* out dtype conversion of fp32 values (ORC_F32 / ORC_F16 / ORC_BF16) */
static void store_as(int ot, void *out, int64_t idx, float v) {
    if (ot == ORC_F32) ((float *)out)[idx] = v;
    else if (ot == ORC_F16) ((uint16_t *)out)[idx] = orc_f32_to_f16(v);
    else ((uint16_t *)out)[idx] = orc_f32_to_bf16(v);
}

int orc_dequantize(int type, const uint8_t *w, int64_t rows, int64_t k, void *out, int ot) {
    int64_t rs = orc_row_size(type, k);
    if (rs < 0) return -1;
    float *tmp = (float *)malloc(sizeof(float) * (size_t)k);
    for (int64_t r = 0; r < rows; r++) {
        orc_dequantize_row(type, w + r * rs, k, tmp);
        for (int64_t i = 0; i < k; i++) store_as(ot, out, r * k + i, tmp[i]);
    }
    free(tmp);
    return 0;
}

/* out[i, :] = dequant(table[ids[i], :]); ids outside [0, rows) leave the row at 0 */
int orc_get_rows(int type, const uint8_t *table, int64_t rows, int64_t k, const int32_t *ids, int64_t n_ids,
                 void *out, int ot) {
    int64_t rs = orc_row_size(type, k);
    if (rs < 0) return -1;
    float *tmp = (float *)malloc(sizeof(float) * (size_t)k);
    for (int64_t i = 0; i < n_ids; i++) {
        int64_t id = ids[i];
        if (id < 0 || id >= rows) {
            for (int64_t c = 0; c < k; c++) store_as(ot, out, i * k + c, 0.0f);
            continue;
        }
        orc_dequantize_row(type, table + id * rs, k, tmp);
        for (int64_t c = 0; c < k; c++) store_as(ot, out, i * k + c, tmp[c]);
    }
    free(tmp);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* per-block integer dot products                                           */
/* ------------------------------------------------------------------------ */

/* S for sub-block j of weight block wb against the q8_1 activation row xq
 * (the row's blocks of 32, indexed from the weight block's first value).     */
static int32_t block_dot(int type, const uint8_t *wb, int64_t first, const uint8_t *xq, int j) {
    int64_t sub = orc_sub_elems(type);
    int32_t S = 0;
    for (int64_t t = 0; t < sub; t++) {
        int i = (int)(j * sub + t);       /* index inside the weight block */
        int64_t kk = first + i;           /* index along K */
        const uint8_t *ab = xq + (kk / 32) * 36;
        int qa = q8_1_q(ab, (int)(kk % 32));
        int qw;
        switch (type) {
        case ORC_Q8_0: qw = q8_0_q(wb, i); break;
        case ORC_Q4_0: qw = q4_0_q(wb, i) - 8; break;
        case ORC_MXFP4: qw = mxfp4_q(wb, i); break;
        case ORC_Q4_1: qw = q4_1_q(wb, i); break;
        case ORC_Q5_0: qw = q5_0_q(wb, i) - 16; break;
        case ORC_Q5_1: qw = q5_1_q(wb, i); break;
        case ORC_Q4_K: qw = q4_k_q(wb, i); break;
        case ORC_Q5_K: qw = q5_k_q(wb, i); break;
        case ORC_Q6_K: qw = q6_k_q(wb, i) - 32; break;
        default: qw = 0;
        }
        S += qw * qa;
    }
    return S;
}

/* sums[m][n][k / sub]: the int32 dot of every weight sub-block with the
 * matching 16 or 32 activation quants. */
int orc_block_dots(int type, const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, int32_t *sums) {
    int64_t rs = orc_row_size(type, k), sub = orc_sub_elems(type);
    if (rs < 0 || sub == 0) return -1;
    int64_t be = orc_block_elems(type), bb = orc_block_bytes(type);
    int64_t nsub = k / sub, xrs = k / 32 * 36;
    for (int64_t r = 0; r < m; r++)
        for (int64_t c = 0; c < n; c++)
            for (int64_t s = 0; s < nsub; s++) {
                int64_t b = s * sub / be;
                int j = (int)(s - b * (be / sub));
                sums[(r * n + c) * nsub + s] = block_dot(type, w + c * rs + b * bb, b * be, xq + r * xrs, j);
            }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* matmul reference: blockwise formula in fp64                               */
/* ------------------------------------------------------------------------ */

/* y = sum over the row's sub-blocks of the combination of stored fields:
 *   Q8_0, Q4_0: d_w * d_a * S      (Q4_0: S over q - 8)
 *   MXFP4:      2^(e - 128) * d_a * S   (S over 2 * e2m1(q))
 *   Q5_0:       d_w * d_a * S           (S over q - 16)
 *   Q4_1, Q5_1: d * d_a * S + m * s_a
 *   Q4_K, Q5_K: d * s_j * d_a * S_j - dmin * m_j * s_a
 *   Q6_K: d * sc_j * d_a * S_j
 * with d_a, s_a the q8_1 fields of the 32-block holding sub-block j.         */
static double dot_row(int type, const uint8_t *wrow, int64_t k, const uint8_t *xrow) {
    int64_t be = orc_block_elems(type), bb = orc_block_bytes(type), sub = orc_sub_elems(type);
    double y = 0.0;
    for (int64_t b = 0; b < k / be; b++) {
        const uint8_t *wb = wrow + b * bb;
        for (int j = 0; j < be / sub; j++) {
            int64_t kk = b * be + j * sub;
            const uint8_t *ab = xrow + (kk / 32) * 36;
            double da = q8_1_d(ab), sa = q8_1_s(ab);
            double S = block_dot(type, wb, b * be, xrow, j);
            if (type == ORC_Q8_0) {
                y += (double)q8_0_d(wb) * da * S;
            } else if (type == ORC_Q4_0) {
                y += (double)q4_0_d(wb) * da * S;
            } else if (type == ORC_MXFP4) {
                y += ldexp(1.0, mxfp4_e(wb) - 128) * da * S;
            } else if (type == ORC_Q5_0) {
                y += (double)q5_0_d(wb) * da * S;
            } else if (type == ORC_Q4_1 || type == ORC_Q5_1) {
                y += (double)q41_d(wb) * da * S + (double)q41_m(wb) * sa;
            } else if (type == ORC_Q4_K || type == ORC_Q5_K) {
                int s, m;
                q4_k_scale_min(wb, j, &s, &m);
                y += (double)q4_k_d(wb) * s * da * S - (double)q4_k_dmin(wb) * m * sa;
            } else {
                y += (double)q6_k_d(wb) * q6_k_scale(wb, j * 16) * da * S;
            }
        }
    }
    return y;
}

struct mm_job {
    int type;
    const uint8_t *w;
    int64_t n, k;
    const uint8_t *xq;
    int64_t m;
    double *y;
    int64_t n0, n1;
};

static void *mm_worker(void *arg) {
    struct mm_job *j = (struct mm_job *)arg;
    int64_t rs = orc_row_size(j->type, j->k), xrs = j->k / 32 * 36;
    for (int64_t c = j->n0; c < j->n1; c++)
        for (int64_t r = 0; r < j->m; r++)
            j->y[r * j->n + c] = dot_row(j->type, j->w + c * rs, j->k, j->xq + r * xrs);
    return NULL;
}

/* y[m][n] (fp64) for weight rows [n0, n1) only; other entries untouched.
 * nthreads > 1 splits the rows over POSIX threads (plain row split).        */
int orc_mul_mat_rows(int type, const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, double *y,
                     int64_t n0, int64_t n1, int nthreads) {
    if (orc_row_size(type, k) < 0 || orc_sub_elems(type) == 0 || k % 32) return -1;
    if (n0 < 0 || n1 > n || n0 > n1) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    struct mm_job jobs[256];
    pthread_t th[256];
    int64_t span = n1 - n0;
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (struct mm_job){type, w, n, k, xq, m, y, n0 + span * t / nthreads, n0 + span * (t + 1) / nthreads};
        if (nthreads == 1) mm_worker(&jobs[t]);
        else pthread_create(&th[t], NULL, mm_worker, &jobs[t]);
    }
    if (nthreads > 1)
        for (int t = 0; t < nthreads; t++) pthread_join(th[t], NULL);
    return 0;
}

int orc_mul_mat(int type, const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, double *y) {
    return orc_mul_mat_rows(type, w, n, k, xq, m, y, 0, n, 1);
}

/* Closed form used to pin the blockwise formula: the plain fp64 dot product of
 * the dequantized weight row with the dequantized activation row.            */
int orc_mul_mat_dequant_f64(int type, const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m,
                            double *y) {
    int64_t rs = orc_row_size(type, k);
    if (rs < 0 || k % 32) return -1;
    double *wr = (double *)malloc(sizeof(double) * (size_t)k);
    double *xr = (double *)malloc(sizeof(double) * (size_t)k);
    for (int64_t c = 0; c < n; c++) {
        orc_dequantize_row_f64(type, w + c * rs, k, wr);
        for (int64_t r = 0; r < m; r++) {
            orc_dequantize_row_f64(ORC_Q8_1, xq + r * (k / 32 * 36), k, xr);
            double acc = 0.0;
            for (int64_t i = 0; i < k; i++) acc += wr[i] * xr[i];
            y[r * n + c] = acc;
        }
    }
    free(wr);
    free(xr);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* MoE: mul_mat_id gate_up -> SwiGLU -> bf16 -> q8_1 -> mul_mat_id down      */
/*      -> expert-weighted sum                                               */
/* ------------------------------------------------------------------------ */

/* Expert e's packed [rows, k] matrix starts at bank + e * stride bytes.  The
 * gate rows come first (0 .. I-1), then the up rows (I .. 2I-1), as a merged
 * gate_up tensor is laid out (transformers PR #45977, "GgufExperts" restructure). */

struct moe_gu_job {
    int wt; const uint8_t *bank; int64_t stride, two_i, h;
    const uint8_t *xq; const int32_t *ids; int64_t n_routes, top_k, n_experts;
    float *hbuf; uint8_t *hq; int64_t r0, r1;
};

static double silu_f64(double z) { return z / (1.0 + exp(-z)); }

static void *moe_gu_worker(void *arg) {
    struct moe_gu_job *j = (struct moe_gu_job *)arg;
    int64_t I = j->two_i / 2;
    int64_t rs = orc_row_size(j->wt, j->h), xrs = j->h / 32 * 36, hrs = I / 32 * 36;
    float *hrow = (float *)malloc(sizeof(float) * (size_t)I);
    for (int64_t r = j->r0; r < j->r1; r++) {
        int64_t t = r / j->top_k;
        int32_t e = j->ids[r];
        if (e < 0 || e >= j->n_experts) {
            for (int64_t i = 0; i < I; i++) hrow[i] = 0.0f;
        } else {
            const uint8_t *we = j->bank + (int64_t)e * j->stride;
            for (int64_t i = 0; i < I; i++) {
                double g = dot_row(j->wt, we + i * rs, j->h, j->xq + t * xrs);
                double u = dot_row(j->wt, we + (I + i) * rs, j->h, j->xq + t * xrs);
                /* the intermediate is kept in the activation dtype (bf16): the
                 * fp64 value rounded once, with no fp32 step in between */
                hrow[i] = orc_bf16_to_f32(orc_f64_to_bf16(silu_f64(g) * u));
            }
        }
        if (j->hbuf) memcpy(j->hbuf + r * I, hrow, sizeof(float) * (size_t)I);
        orc_quantize_q8_1(hrow, 1, I, I, j->hq + r * hrs);
    }
    free(hrow);
    return NULL;
}

/* For every route r = t * top_k + kk: h[r] = bf16(silu(g) * u), then q8_1.
 * xq: [n_tokens][h/32] q8_1.  hbuf (optional): [n_routes][I] fp32 copy of the
 * bf16 h.  hq: [n_routes][I/32] q8_1.  Inactive routes (id < 0 or >= E) give h = 0. */
int orc_moe_gate_up(int wt, const uint8_t *bank, int64_t n_experts, int64_t stride, int64_t two_i, int64_t h,
                    const uint8_t *xq, const int32_t *ids, int64_t n_tokens, int64_t top_k, float *hbuf, uint8_t *hq,
                    int64_t r0, int64_t r1, int nthreads) {
    if (two_i % 64 || orc_row_size(wt, h) < 0) return -1;
    int64_t n_routes = n_tokens * top_k;
    if (r1 < 0) r1 = n_routes;
    if (r0 < 0 || r1 > n_routes || r0 > r1) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    struct moe_gu_job jobs[256];
    pthread_t th[256];
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (struct moe_gu_job){wt, bank, stride, two_i, h, xq, ids, n_routes, top_k, n_experts, hbuf, hq,
                                      r0 + (r1 - r0) * t / nthreads, r0 + (r1 - r0) * (t + 1) / nthreads};
        if (nthreads == 1) moe_gu_worker(&jobs[t]);
        else pthread_create(&th[t], NULL, moe_gu_worker, &jobs[t]);
    }
    if (nthreads > 1)
        for (int t = 0; t < nthreads; t++) pthread_join(th[t], NULL);
    return 0;
}

struct moe_dn_job {
    int wt; const uint8_t *bank; int64_t stride, n_out, i_dim;
    const uint8_t *hq; const int32_t *ids; const float *route_w; int64_t top_k, n_experts;
    double *y; int64_t t0, t1;
};

static void *moe_dn_worker(void *arg) {
    struct moe_dn_job *j = (struct moe_dn_job *)arg;
    int64_t rs = orc_row_size(j->wt, j->i_dim), hrs = j->i_dim / 32 * 36;
    for (int64_t t = j->t0; t < j->t1; t++) {
        for (int64_t c = 0; c < j->n_out; c++) j->y[t * j->n_out + c] = 0.0;
        for (int64_t kk = 0; kk < j->top_k; kk++) {
            int64_t r = t * j->top_k + kk;
            int32_t e = j->ids[r];
            if (e < 0 || e >= j->n_experts) continue;
            double wgt = j->route_w ? (double)j->route_w[r] : 1.0;
            if (wgt == 0.0) continue;
            const uint8_t *we = j->bank + (int64_t)e * j->stride;
            for (int64_t c = 0; c < j->n_out; c++)
                j->y[t * j->n_out + c] += wgt * dot_row(j->wt, we + c * rs, j->i_dim, j->hq + r * hrs);
        }
    }
    return NULL;
}

/* y[t] = sum_kk w[t,kk] * (W_down[ids[t,kk]] . hq[t*top_k + kk]) in fp64, for
 * tokens [t0, t1).  Inactive routes and zero weights contribute nothing.     */
int orc_moe_down(int wt, const uint8_t *bank, int64_t n_experts, int64_t stride, int64_t n_out, int64_t i_dim,
                 const uint8_t *hq, const int32_t *ids, const float *route_w, int64_t n_tokens, int64_t top_k,
                 double *y, int64_t t0, int64_t t1, int nthreads) {
    if (orc_row_size(wt, i_dim) < 0 || i_dim % 32) return -1;
    if (t1 < 0) t1 = n_tokens;
    if (t0 < 0 || t1 > n_tokens || t0 > t1) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    struct moe_dn_job jobs[256];
    pthread_t th[256];
    for (int t = 0; t < nthreads; t++) {
        jobs[t] = (struct moe_dn_job){wt, bank, stride, n_out, i_dim, hq, ids, route_w, top_k, n_experts, y,
                                      t0 + (t1 - t0) * t / nthreads, t0 + (t1 - t0) * (t + 1) / nthreads};
        if (nthreads == 1) moe_dn_worker(&jobs[t]);
        else pthread_create(&th[t], NULL, moe_dn_worker, &jobs[t]);
    }
    if (nthreads > 1)
        for (int t = 0; t < nthreads; t++) pthread_join(th[t], NULL);
    return 0;
}

/* mul_mat_id without the weighted sum: y[r] = W[ids[r]] . xq[r / top_k] for
 * every route r = t * top_k + j (x rows per token, shared by the token's
 * routes), in fp64; an inactive route (id < 0 or >= E) gives a zero row.    */
int orc_moe_plain(int wt, const uint8_t *bank, int64_t n_experts, int64_t stride, int64_t n, int64_t k,
                  const uint8_t *xq, const int32_t *ids, int64_t n_tokens, int64_t top_k, double *y) {
    int64_t rs = orc_row_size(wt, k), xrs = k / 32 * 36;
    if (rs < 0 || k % 32) return -1;
    for (int64_t r = 0; r < n_tokens * top_k; r++) {
        int32_t e = ids[r];
        for (int64_t c = 0; c < n; c++) {
            if (e < 0 || e >= n_experts) {
                y[r * n + c] = 0.0;
                continue;
            }
            y[r * n + c] = dot_row(wt, bank + (int64_t)e * stride + c * rs, k, xq + (r / top_k) * xrs);
        }
    }
    return 0;
}
