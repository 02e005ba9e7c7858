// dequantize / get_rows / float conversion / per-block int32 dot sums.
//
// dequantize and get_rows are the ops of the same names in FreeToken PR #690
// "serve GGUF checkpoints on vendored ggml-cuda kernels" (section "Vendored
// ggml", paragraph "Our own code next to it").  Values are computed in fp32 in
// the order  Q4_K, Q5_K: a = d*s; b = dmin*m; a*q - b;  Q6_K: (d*sc)*(q-32);
// Q8_0 / q8_1: d*q;  Q4_0: d*(q-8);  MXFP4: +-(2^(e-128) * |2 e2m1(q)|)  and
// rounded to the output dtype (RNE).
// Every product above is exact in fp32, so the only rounding is the Q4_K /
// Q5_K subtraction.
//
// One thread produces one 32-value piece of a row:
//   Q8_0 / q8_1 / Q4_0 / MXFP4 : one block (one run of 32 values)
//   Q4_K / Q5_K : sub-block j of a super-block (values [32j, +32): the low or
//                 high nibbles of the 32 quant bytes of chunk j / 2; Q5_K adds
//                 bit j of the 32 high-bit bytes)
//   Q6_K        : runs [128h + 32g + l0, +8) for g = 0..3 of a super-block
#include "common.cuh"
#include "internal.h"

namespace gg {

template <int OT>
__device__ __forceinline__ void store_run(void *out, int64_t off, const float *v, int n) {
    // n is 8, 16 or 32; off is a multiple of 8 values
    if (OT == GGUF_F32) {
        float4 *p = reinterpret_cast<float4 *>(reinterpret_cast<float *>(out) + off);
        for (int i = 0; i < n / 4; i++) p[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
    } else {
        uint4 *p = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(out) + off);
        for (int i = 0; i < n / 8; i++) {
            uint32_t w[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                float a = v[8 * i + 2 * j], b = v[8 * i + 2 * j + 1];
                uint16_t ha = OT == GGUF_BF16 ? f2bf_rn(a) : f2h_rn(a);
                uint16_t hb = OT == GGUF_BF16 ? f2bf_rn(b) : f2h_rn(b);
                w[j] = (uint32_t)ha | ((uint32_t)hb << 16);
            }
            p[i] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

template <int WT, int OT>
__global__ void __launch_bounds__(256) dequant_kernel(const uint8_t *__restrict__ w, int64_t rows, int64_t k,
                                                      int64_t rb, const int32_t *__restrict__ ids,
                                                      int64_t table_rows, void *__restrict__ out) {
    const int64_t P = k / 32;
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= rows * P) return;
    const int64_t r = g / P;
    const int64_t p = g - r * P;
    int64_t src = r;
    bool zero = false;
    if (ids != nullptr) {
        const int64_t id = ids[r];
        zero = id < 0 || id >= table_rows;
        src = zero ? 0 : id;
    }
    const uint8_t *row = w + src * rb;
    const int64_t obase = r * k;
    float v[32];
    if (WT == GGUF_Q8_0 || WT == GGUF_Q8_1) {
        const int bb = WT == GGUF_Q8_0 ? Q8_0_BYTES : Q8_1_BYTES;
        const uint8_t *blk = row + p * bb;
        const float d = h2f(ld_u16(blk));
        const uint8_t *q = blk + (WT == GGUF_Q8_0 ? 2 : 4);
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const uint16_t two = ld_u16(q + 2 * i);
            v[2 * i] = __fmul_rn(d, (float)(int8_t)(two & 0xff));
            v[2 * i + 1] = __fmul_rn(d, (float)(int8_t)(two >> 8));
        }
        if (zero) for (int i = 0; i < 32; i++) v[i] = 0.0f;
        store_run<OT>(out, obase + p * 32, v, 32);
    } else if (WT == GGUF_Q4_0) {
        // block p: byte l of the 16 quant bytes holds value l (low nibble) and
        // value l + 16 (high nibble); blocks are only 2-byte aligned
        const uint8_t *blk = row + p * Q4_0_BYTES;
        const float d = h2f(ld_u16(blk));
        uint32_t qw[4];
        ldw_a2<4>(blk + 2, qw);
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const int byte = (int)((qw[i >> 2] >> (8 * (i & 3))) & 0xff);
            v[i] = __fmul_rn(d, (float)((byte & 15) - 8));
            v[16 + i] = __fmul_rn(d, (float)((byte >> 4) - 8));
        }
        if (zero) for (int i = 0; i < 32; i++) v[i] = 0.0f;
        store_run<OT>(out, obase + p * 32, v, 32);
    } else if (WT == GGUF_MXFP4) {
        // block p (17 bytes, any alignment): e2m1 code of value l in the low
        // nibble of code byte l, of value l + 16 in the high one
        uint32_t e, qw[4];
        ld_mxfp4_block(row + p * MXFP4_BYTES, e, qw);
        const float d = e8m0_half(e);
#pragma unroll
        for (int i = 0; i < 16; i++) {
            const uint32_t byte = (qw[i >> 2] >> (8 * (i & 3))) & 0xff;
            const int k0 = mxfp4_k(byte & 15), k1 = mxfp4_k(byte >> 4);
            const float a0 = __fmul_rn(d, (float)(k0 < 0 ? -k0 : k0)), a1 = __fmul_rn(d, (float)(k1 < 0 ? -k1 : k1));
            v[i] = (byte & 8) ? -a0 : a0;
            v[16 + i] = (byte & 0x80) ? -a1 : a1;
        }
        if (zero) for (int i = 0; i < 32; i++) v[i] = 0.0f;
        store_run<OT>(out, obase + p * 32, v, 32);
    } else if (WT == GGUF_Q4_K || WT == GGUF_Q5_K) {
        // sub-block j = p % 8 of super-block p / 8: the low (j even) or high
        // (j odd) nibbles of the 32 quant bytes of chunk j / 2 (Q5_K: plus bit
        // j of the 32 high-bit bytes as the fifth bit), written as one
        // contiguous run of 32 values
        constexpr bool K5 = WT == GGUF_Q5_K;
        const int64_t sb = p >> 3;
        const int j = (int)(p & 7), c = j >> 1, sh = 4 * (j & 1);
        const uint8_t *blk = row + sb * (K5 ? Q5_K_BYTES : Q4_K_BYTES);
        const int qoff = K5 ? 48 : 16;
        const uint4 hdr = *reinterpret_cast<const uint4 *>(blk);
        const uint4 q0 = *reinterpret_cast<const uint4 *>(blk + qoff + 32 * c);
        const uint4 q1 = *reinterpret_cast<const uint4 *>(blk + qoff + 16 + 32 * c);
        uint4 h0 = make_uint4(0u, 0u, 0u, 0u), h1 = h0;
        if (K5) {
            h0 = *reinterpret_cast<const uint4 *>(blk + 16);
            h1 = *reinterpret_cast<const uint4 *>(blk + 32);
        }
        const uint32_t sc[3] = {hdr.y, hdr.z, hdr.w};
        const float d = h2f(hdr.x & 0xffff), dmin = h2f(hdr.x >> 16);
        int s, m;
        q4k_scale_min(sc, j, s, m);
        const float a = __fmul_rn(d, (float)s), b = __fmul_rn(dmin, (float)m);
        const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
        const uint32_t hw[8] = {h0.x, h0.y, h0.z, h0.w, h1.x, h1.y, h1.z, h1.w};
#pragma unroll
        for (int i = 0; i < 32; i++) {
            int q = (qw[i >> 2] >> (8 * (i & 3) + sh)) & 15;
            if (K5) q |= (int)((hw[i >> 2] >> (8 * (i & 3) + j)) & 1) << 4;
            v[i] = __fsub_rn(__fmul_rn(a, (float)q), b);
        }
        if (zero) for (int i = 0; i < 32; i++) v[i] = 0.0f;
        store_run<OT>(out, obase + sb * 256 + 32 * j, v, 32);
    } else {  // Q6_K
        const int64_t sb = p >> 3;
        const int pp = (int)(p & 7), h = pp >> 2, l0 = 8 * (pp & 3);
        const uint8_t *blk = row + sb * Q6_K_BYTES;
        uint32_t A[2], B[2], H[2], S[2];
        ld8_a2(blk + 64 * h + l0, A[0], A[1]);
        ld8_a2(blk + 64 * h + 32 + l0, B[0], B[1]);
        ld8_a2(blk + 128 + 32 * h + l0, H[0], H[1]);
        ld8_a2(blk + 192 + 8 * h, S[0], S[1]);
        const float d = h2f(ld_u16(blk + 208));
#pragma unroll
        for (int g4 = 0; g4 < 4; g4++) {
            const int si = (l0 >> 4) + 2 * g4;  // scale byte inside this half's 8
            const int sc = (int)(int8_t)((S[si >> 2] >> (8 * (si & 3))) & 0xff);
            const float dsc = __fmul_rn(d, (float)sc);
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const uint32_t a = (A[i >> 2] >> (8 * (i & 3))) & 0xff;
                const uint32_t b = (B[i >> 2] >> (8 * (i & 3))) & 0xff;
                const uint32_t hb = (H[i >> 2] >> (8 * (i & 3))) & 0xff;
                const uint32_t lo = g4 == 0 ? (a & 15) : g4 == 1 ? (b & 15) : g4 == 2 ? (a >> 4) : (b >> 4);
                const int q = (int)(lo | (((hb >> (2 * g4)) & 3) << 4));
                v[8 * g4 + i] = __fmul_rn(dsc, (float)(q - 32));
            }
        }
        if (zero) for (int i = 0; i < 32; i++) v[i] = 0.0f;
#pragma unroll
        for (int g4 = 0; g4 < 4; g4++) store_run<OT>(out, obase + sb * 256 + 128 * h + 32 * g4 + l0, v + 8 * g4, 8);
    }
}

template <int XT, int OT>
__global__ void convert_kernel(const void *__restrict__ x, int64_t count, void *__restrict__ out) {
    const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= count) return;
    float v;
    if (XT == GGUF_F32) v = reinterpret_cast<const float *>(x)[i];
    else if (XT == GGUF_BF16) v = bf2f(reinterpret_cast<const uint16_t *>(x)[i]);
    else v = h2f(reinterpret_cast<const uint16_t *>(x)[i]);
    store_out(out, OT, i, v);
}

template <int WT>
__global__ void block_dots_kernel(const uint8_t *__restrict__ w, int64_t n, int64_t k, int64_t rb,
                                  const uint8_t *__restrict__ xq, int64_t m, int32_t *__restrict__ sums) {
    constexpr int SUB = WT == GGUF_Q6_K ? 16 : 32;
    const int64_t nsub = k / SUB;
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (g >= m * n * nsub) return;
    const int64_t s = g % nsub;
    const int64_t c = (g / nsub) % n;
    const int64_t r = g / (nsub * n);
    const uint8_t *row = w + c * rb;
    const uint8_t *xrow = xq + r * (k / 32) * Q8_1_BYTES;
    int acc = 0;
    for (int t = 0; t < SUB; t++) {
        const int64_t kk = s * SUB + t;  // position along K
        const int qa = (int8_t)xrow[(kk / 32) * Q8_1_BYTES + 4 + (kk % 32)];
        int qw;
        if (WT == GGUF_Q8_0) {
            qw = (int8_t)row[(kk / 32) * Q8_0_BYTES + 2 + (kk % 32)];
        } else if (WT == GGUF_Q4_0) {
            const uint8_t byte = row[(kk / 32) * Q4_0_BYTES + 2 + (kk % 16)];
            qw = ((kk % 32) < 16 ? (byte & 15) : (byte >> 4)) - 8;
        } else if (WT == GGUF_MXFP4) {
            const uint8_t byte = row[(kk / 32) * MXFP4_BYTES + 1 + (kk % 16)];
            qw = mxfp4_k((kk % 32) < 16 ? (byte & 15) : (byte >> 4));
        } else if (WT == GGUF_Q4_K || WT == GGUF_Q5_K) {
            constexpr bool K5 = WT == GGUF_Q5_K;
            const uint8_t *blk = row + (kk / 256) * (K5 ? Q5_K_BYTES : Q4_K_BYTES);
            const int i = (int)(kk % 256), cc = i / 64, rr = i % 64;
            const uint8_t byte = blk[(K5 ? 48 : 16) + 32 * cc + (rr % 32)];
            qw = rr < 32 ? (byte & 15) : (byte >> 4);
            if (K5) qw |= ((blk[16 + (i % 32)] >> (i / 32)) & 1) << 4;
        } else {
            const uint8_t *blk = row + (kk / 256) * Q6_K_BYTES;
            const int i = (int)(kk % 256), h = i / 128, o = i % 128, l = o % 32, g4 = o / 32;
            const uint8_t *ql = blk + 64 * h, *qh = blk + 128 + 32 * h;
            const int lo = g4 == 0 ? (ql[l] & 15) : g4 == 1 ? (ql[l + 32] & 15) : g4 == 2 ? (ql[l] >> 4) : (ql[l + 32] >> 4);
            qw = (lo | (((qh[l] >> (2 * g4)) & 3) << 4)) - 32;
        }
        acc += qw * qa;
    }
    sums[g] = acc;
}

cudaError_t launch_dequantize(const uint8_t *w, int wt, int64_t rows, int64_t k, const int32_t *ids,
                              int64_t table_rows, void *out, int ot, cudaStream_t s) {
    const int64_t threads = rows * (k / 32);
    if (threads == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((threads + 255) / 256);
    const int64_t rb = k / block_elems(wt) * block_bytes(wt);
#define DQ(WT, OT) dequant_kernel<WT, OT><<<grid, 256, 0, s>>>(w, rows, k, rb, ids, table_rows, out)
#define DQT(WT) do { if (ot == GGUF_F32) DQ(WT, GGUF_F32); else if (ot == GGUF_BF16) DQ(WT, GGUF_BF16); else DQ(WT, GGUF_F16); } while (0)
    switch (wt) {
    case GGUF_Q8_0: DQT(GGUF_Q8_0); break;
    case GGUF_Q8_1: DQT(GGUF_Q8_1); break;
    case GGUF_Q4_0: DQT(GGUF_Q4_0); break;
    case GGUF_Q4_K: DQT(GGUF_Q4_K); break;
    case GGUF_Q5_K: DQT(GGUF_Q5_K); break;
    case GGUF_MXFP4: DQT(GGUF_MXFP4); break;
    case GGUF_Q6_K: DQT(GGUF_Q6_K); break;
    default: return cudaErrorInvalidValue;
    }
#undef DQT
#undef DQ
    return cudaGetLastError();
}

cudaError_t launch_convert_float(const void *x, int xt, int64_t count, void *out, int ot, cudaStream_t s) {
    if (count == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((count + 255) / 256);
#define CV(XT, OT) convert_kernel<XT, OT><<<grid, 256, 0, s>>>(x, count, out)
#define CVT(XT) do { if (ot == GGUF_F32) CV(XT, GGUF_F32); else if (ot == GGUF_BF16) CV(XT, GGUF_BF16); else CV(XT, GGUF_F16); } while (0)
    if (xt == GGUF_F32) CVT(GGUF_F32);
    else if (xt == GGUF_BF16) CVT(GGUF_BF16);
    else CVT(GGUF_F16);
#undef CVT
#undef CV
    return cudaGetLastError();
}

cudaError_t launch_block_dots(const uint8_t *w, int wt, int64_t n, int64_t k, const uint8_t *xq, int64_t m,
                              int32_t *sums, cudaStream_t s) {
    const int sub = wt == GGUF_Q6_K ? 16 : 32;
    const int64_t threads = m * n * (k / sub);
    if (threads == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((threads + 255) / 256);
    const int64_t rb = k / block_elems(wt) * block_bytes(wt);
    switch (wt) {
    case GGUF_Q8_0: block_dots_kernel<GGUF_Q8_0><<<grid, 256, 0, s>>>(w, n, k, rb, xq, m, sums); break;
    case GGUF_Q4_0: block_dots_kernel<GGUF_Q4_0><<<grid, 256, 0, s>>>(w, n, k, rb, xq, m, sums); break;
    case GGUF_Q4_K: block_dots_kernel<GGUF_Q4_K><<<grid, 256, 0, s>>>(w, n, k, rb, xq, m, sums); break;
    case GGUF_Q5_K: block_dots_kernel<GGUF_Q5_K><<<grid, 256, 0, s>>>(w, n, k, rb, xq, m, sums); break;
    case GGUF_MXFP4: block_dots_kernel<GGUF_MXFP4><<<grid, 256, 0, s>>>(w, n, k, rb, xq, m, sums); break;
    case GGUF_Q6_K: block_dots_kernel<GGUF_Q6_K><<<grid, 256, 0, s>>>(w, n, k, rb, xq, m, sums); break;
    default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

}  // namespace gg
