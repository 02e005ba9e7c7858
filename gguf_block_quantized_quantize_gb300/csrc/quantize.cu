// q8_1 activation quantization (FreeToken PR #690 "serve GGUF checkpoints on
// vendored ggml-cuda kernels", section "Vendored ggml": fp32 / bf16 / fp16
// activations go straight to q8_1).
//
// One thread handles 8 consecutive values, four threads one block of 32:
//   d = amax / 127 (IEEE division), q = roundf(x / d) (ties away from zero),
//   s = fp16(d * sum(q)) with the fp32 d, and d is stored as fp16(d).
// The kernel is HBM-bound: 2 or 4 bytes read and 1.125 bytes written per value.
#include "common.cuh"
#include "internal.h"

namespace gg {

template <int XT, bool VEC>
__device__ __forceinline__ void load8(const void *x, int64_t off, float v[8]) {
    if (XT == GGUF_F32) {
        const float *p = reinterpret_cast<const float *>(x) + off;
        if (VEC) {
            float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
            v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
        } else {
#pragma unroll
            for (int i = 0; i < 8; i++) v[i] = p[i];
        }
    } else {
        const uint16_t *p = reinterpret_cast<const uint16_t *>(x) + off;
        uint16_t h[8];
        if (VEC) {
            uint4 a = *reinterpret_cast<const uint4 *>(p);
            uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int i = 0; i < 4; i++) { h[2 * i] = w[i] & 0xffff; h[2 * i + 1] = w[i] >> 16; }
        } else {
#pragma unroll
            for (int i = 0; i < 8; i++) h[i] = p[i];
        }
#pragma unroll
        for (int i = 0; i < 8; i++) v[i] = (XT == GGUF_BF16) ? bf2f(h[i]) : h2f(h[i]);
    }
}

// fp16 tensor-core operand of 8 q8_1 values: hi = fp16(d16 * q) (d16 * q is
// exact in fp32), and optionally lo = fp16(d16 * q - hi), which makes hi + lo
// equal to d16 * q (the 3-term product of the precise mode needs it).
__device__ __forceinline__ void write_f16_operand(float d16, const int q[8], uint16_t *hi, uint16_t *lo) {
    uint32_t hw[4], lw[4];
#pragma unroll
    for (int i = 0; i < 4; i++) {
        const float v0 = d16 * (float)q[2 * i], v1 = d16 * (float)q[2 * i + 1];
        const uint16_t h0 = f2h_rn(v0), h1 = f2h_rn(v1);
        hw[i] = (uint32_t)h0 | ((uint32_t)h1 << 16);
        lw[i] = (uint32_t)f2h_rn(v0 - h2f(h0)) | ((uint32_t)f2h_rn(v1 - h2f(h1)) << 16);
    }
    *reinterpret_cast<uint4 *>(hi) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    if (lo) *reinterpret_cast<uint4 *>(lo) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
}

// Min-term correction columns of the operand rows (Q4_K / Q5_K weights).  The fp16
// operand d16 * q gives the min term of a 32-block as dmin * m * d16 * sum(q);
// the blockwise formula uses the stored s instead.  Column k + b of a row
// holds c_b = d16 * sum(q) - s (the weight side holds dmin * m for that
// sub-block), so the product adds exactly the difference.  Columns past
// k + k/32 up to the row pitch are zero, and so are all low parts there.
__device__ __forceinline__ void write_correction(uint16_t *hi_row, uint16_t *lo_row, int64_t k, int64_t pitch,
                                                 int64_t b, int j, float d16, int sum, uint16_t s16) {
    const int64_t nb = k / QK8;
    if (j == 0) hi_row[k + b] = f2h_rn(d16 * (float)sum - h2f(s16));
    if (j == 1 && lo_row) lo_row[k + b] = 0;
    // zero padding [k + nb, pitch): column k + nb + 4 * b + j, then every 4 * nb
    for (int64_t c = k + nb + 4 * b + j; c < pitch; c += 4 * nb) {
        hi_row[c] = 0;
        if (lo_row) lo_row[c] = 0;
    }
}

// Scatter of the permuted operand (MoE): input row i feeds the routes
// r = i * fan + j (j < fan); an active route (pos[r] >= 0) is written to row
// offsets[ids[r]] + pos[r] of the output (grouped route order), a skipped one
// nowhere.  ids == nullptr: output row i is input row i.
struct RowScatter {
    const int32_t *ids, *pos, *offsets;
    int32_t fan;
};

// the fp16 operand row(s) of one 8-value group: row i, or every active
// route's grouped row
__device__ __forceinline__ void write_operand_rows(const RowScatter &map, int64_t row, int64_t k, int64_t pitch,
                                                   int64_t b, int j, float d16, const int q[8], int sum,
                                                   uint16_t s16, uint16_t *xh, uint16_t *xl) {
    for (int f = 0; f < (map.ids ? map.fan : 1); f++) {
        int64_t orow = row;
        if (map.ids) {
            const int64_t r = row * map.fan + f;
            const int32_t pr = map.pos[r];
            if (pr < 0) continue;
            orow = (int64_t)map.offsets[map.ids[r]] + pr;
        }
        write_f16_operand(d16, q, xh + orow * pitch + b * QK8 + 8 * j, xl ? xl + orow * pitch + b * QK8 + 8 * j : nullptr);
        if (pitch > k)
            write_correction(xh + orow * pitch, xl ? xl + orow * pitch : nullptr, k, pitch, b, j, d16, sum, s16);
    }
}

template <int XT, bool VEC>
__global__ void __launch_bounds__(256) quantize_q8_1_kernel(const void *__restrict__ x, int64_t m, int64_t k,
                                                            int64_t ldx, uint8_t *__restrict__ xq,
                                                            uint16_t *__restrict__ xh, uint16_t *__restrict__ xl,
                                                            int64_t pitch, RowScatter map, RouteMarks mk) {
    // launched as a programmatic dependent: let the next kernel start its own
    // independent prefetch, and wait for the previous kernel before touching
    // memory it may still read or write
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t nb = k / QK8;
    const int64_t total = m * nb;
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (mk.ids != nullptr && g < mk.R) {   // the MoE route marks (see RouteMarks)
        const int32_t e = mk.ids[g];
        const bool ok = e >= 0 && e < mk.E && !(mk.skip_zero_w && mk.rw != nullptr && mk.rw[g] == 0.0f);
        if (e >= mk.E && mk.status != nullptr) atomicAdd(mk.status, 1);
        mk.pos[g] = ok ? (int32_t)g : -1;
    }
    const int64_t blk = g >> 2;
    const int j = (int)(g & 3);
    const bool active = blk < total;
    const int64_t row = active ? blk / nb : 0;
    const int64_t b = active ? blk - row * nb : 0;

    float v[8];
    if (active) load8<XT, VEC>(x, row * ldx + b * QK8 + 8 * j, v);
    else {
#pragma unroll
        for (int i = 0; i < 8; i++) v[i] = 0.0f;
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; i++) amax = fmaxf(amax, fabsf(v[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const float d = __fdiv_rn(amax, 127.0f);

    int q[8];
    int sum = 0;
#pragma unroll
    for (int i = 0; i < 8; i++) {
        q[i] = (d != 0.0f) ? (int)roundf(__fdiv_rn(v[i], d)) : 0;
        sum += q[i];
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    if (!active) return;

    const uint16_t dh = f2h_rn(d);
    if (xq != nullptr) {
        uint8_t *o = xq + blk * Q8_1_BYTES;
        uint32_t w0 = (q[0] & 0xff) | ((q[1] & 0xff) << 8) | ((q[2] & 0xff) << 16) | ((uint32_t)(q[3] & 0xff) << 24);
        uint32_t w1 = (q[4] & 0xff) | ((q[5] & 0xff) << 8) | ((q[6] & 0xff) << 16) | ((uint32_t)(q[7] & 0xff) << 24);
        reinterpret_cast<uint32_t *>(o + 4 + 8 * j)[0] = w0;
        reinterpret_cast<uint32_t *>(o + 4 + 8 * j)[1] = w1;
        if (j == 0) {
            const uint16_t sh = f2h_rn(__fmul_rn(d, (float)sum));
            *reinterpret_cast<uint32_t *>(o) = (uint32_t)dh | ((uint32_t)sh << 16);
        }
    }
    if (xh != nullptr)
        write_operand_rows(map, row, k, pitch, b, j, h2f(dh), q, sum, f2h_rn(__fmul_rn(d, (float)sum)), xh, xl);
}

__global__ void __launch_bounds__(256) q8_1_to_f16_kernel(const uint8_t *__restrict__ xq, int64_t m, int64_t k,
                                                          uint16_t *__restrict__ xh, uint16_t *__restrict__ xl,
                                                          int64_t pitch, RowScatter map) {
    const int64_t nb = k / QK8;
    const int64_t g = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int64_t blk = g >> 2;
    const int j = (int)(g & 3);
    if (blk >= m * nb) return;
    const uint8_t *p = xq + blk * Q8_1_BYTES;
    const float d16 = h2f(ld_u16(p));
    const uint32_t w0 = ld_u32(p + 4 + 8 * j), w1 = ld_u32(p + 8 + 8 * j);
    int q[8];
#pragma unroll
    for (int i = 0; i < 4; i++) { q[i] = (int8_t)(w0 >> (8 * i)); q[4 + i] = (int8_t)(w1 >> (8 * i)); }
    const int64_t row = blk / nb, b = blk - row * nb;
    int sum = 0;
    if (pitch > k)
        for (int t = 0; t < 32; t++) sum += (int8_t)p[4 + t];
    write_operand_rows(map, row, k, pitch, b, j, d16, q, sum, ld_u16(p + 2), xh, xl);
}

cudaError_t launch_quantize_q8_1(const void *x, int xt, int64_t m, int64_t k, int64_t ldx, uint8_t *xq,
                                 uint16_t *xh, uint16_t *xl, cudaStream_t s, int64_t pitch, const int32_t *ids,
                                 const int32_t *pos, const int32_t *offsets, int32_t fan, const RouteMarks &marks) {
    if (pitch < k) pitch = k;
    int64_t threads = m * (k / QK8) * 4;
    if (marks.ids != nullptr && marks.R > threads) threads = marks.R;
    if (threads == 0) return cudaSuccess;
    const int64_t grid = (threads + 255) / 256;
    const int esz = xt == GGUF_F32 ? 4 : 2;
    const bool vec = (reinterpret_cast<uintptr_t>(x) % 16 == 0) && ((ldx * esz) % 16 == 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const RowScatter map{ids, pos, offsets, fan < 1 ? 1 : fan};
#define QLAUNCH(XT, V) \
    (void)cudaLaunchKernelEx(&cfg, quantize_q8_1_kernel<XT, V>, x, m, k, ldx, xq, xh, xl, pitch, map, marks)
    if (xt == GGUF_F32) { if (vec) QLAUNCH(GGUF_F32, true); else QLAUNCH(GGUF_F32, false); }
    else if (xt == GGUF_BF16) { if (vec) QLAUNCH(GGUF_BF16, true); else QLAUNCH(GGUF_BF16, false); }
    else { if (vec) QLAUNCH(GGUF_F16, true); else QLAUNCH(GGUF_F16, false); }
#undef QLAUNCH
    return cudaGetLastError();
}

cudaError_t launch_q8_1_to_f16(const uint8_t *xq, int64_t m, int64_t k, uint16_t *xh, uint16_t *xl, cudaStream_t s,
                               int64_t pitch, const int32_t *ids, const int32_t *pos, const int32_t *offsets,
                               int32_t fan) {
    if (pitch < k) pitch = k;
    const int64_t threads = m * (k / QK8) * 4;
    if (threads == 0) return cudaSuccess;
    q8_1_to_f16_kernel<<<(unsigned)((threads + 255) / 256), 256, 0, s>>>(xq, m, k, xh, xl, pitch,
                                                                        RowScatter{ids, pos, offsets, fan < 1 ? 1 : fan});
    return cudaGetLastError();
}

}  // namespace gg
