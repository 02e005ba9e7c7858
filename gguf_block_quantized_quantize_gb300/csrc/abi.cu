// C ABI of libgguf_gb300: argument validation, path dispatch and error
// reporting.  Every entry point validates on the host, returns a status code
// and never aborts; kernels are launched asynchronously on the caller's stream.
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include <map>
#include <mutex>
#include <string>
#include <tuple>

#include "common.cuh"
#include "internal.h"

namespace gg {

static thread_local std::string g_last_error;

static gguf_status fail(gguf_status st, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return st;
}

// for the other translation units of the C ABI
gguf_status report(gguf_status st, const char *msg) {
    g_last_error = msg;
    return st;
}

static gguf_status cuda_status(cudaError_t e, const char *what) {
    if (e == cudaSuccess) return GGUF_OK;
    return fail(GGUF_ERR_CUDA, "%s: CUDA error %d (%s)", what, (int)e, cudaGetErrorString(e));
}

const DeviceInfo &device_info() {
    static DeviceInfo infos[64];
    static bool have[64];
    static std::mutex mu;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    std::lock_guard<std::mutex> lock(mu);
    if (!have[dev]) {
        DeviceInfo di{};
        cudaDeviceGetAttribute(&di.sm_count, cudaDevAttrMultiProcessorCount, dev);
        cudaDeviceGetAttribute(&di.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&di.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
        int optin = 0;
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        di.smem_optin = (size_t)optin;
        if (di.sm_count <= 0) di.sm_count = 1;
        infos[dev] = di;
        have[dev] = true;
    }
    return infos[dev];
}

int kernel_occupancy(const void *kern, int threads, size_t smem, cudaError_t *err) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void *, int, size_t>, int> cache;
    static std::map<std::pair<int, const void *>, size_t> smem_limit;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        *err = e;
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(dev, kern, threads, smem);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
    size_t &lim = smem_limit[std::make_pair(dev, kern)];
    if (smem > lim) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) {
            *err = e;
            return 0;
        }
        lim = smem;
    }
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess) {
        *err = e;
        return 0;
    }
    if (per_sm < 1) per_sm = 1;
    cache[key] = per_sm;
    return per_sm;
}

// tunables
static int64_t g_mmvq_max_m = 8;
static int64_t g_mmq_enable = 1;
static int64_t g_mmvq_tc = 1;
static int64_t g_mmvq_tc_max_m = 16;   // 9..16 tokens: 2 n-tiles beat MMQ; 4 n-tiles do not
static int64_t g_mmvq_tc_min_m = 5;
// MoE calls of at most this many tokens take the route-batched MMVQ (vector)
// path; the workspace reserves its buffers up to MOE_VEC_CAP tokens
constexpr int64_t MOE_VEC_CAP = 256;
static int64_t g_moe_vec_max_tokens = 256;
static int64_t g_mmq_stage = 1;
static int64_t g_moe_deterministic = 1;
static int64_t g_mmq_bn_max = 256;
static int64_t g_mmq_split_k = 1;   // small m: split K across CTAs (fp32 partial sums) to fill the GPU
static int64_t g_mmq_engine = 0;    // 1: 16-bit-output prefill products as dequantize + library GEMM
int64_t option_mmq_engine() { return g_mmq_engine; }
// the library-GEMM engine takes this product
static bool lib_engine(int64_t m, int64_t k, int yt) { return g_mmq_engine == 1 && yt != GGUF_F32 && m > 0 && k > 0; }
int64_t option_mmq_bn_max() { return g_mmq_bn_max; }
static int64_t g_moe_down_precise = 0;
// gate_up GEMM of the grouped MoE path: 1 hi + lo operands (three MMAs per K
// step), 0 one fp16 operand per side
static int64_t g_moe_gate_up_precise = 1;
int64_t option_mmq_stage() { return g_mmq_stage; }
int64_t option_moe_deterministic() { return g_moe_deterministic; }
int64_t option_mmvq_tc() { return g_mmvq_tc; }
int64_t option_mmvq_tc_min_m() { return g_mmvq_tc_min_m; }
int64_t option_mmvq_tc_max_m() { return g_mmvq_tc_max_m; }

static bool is_float(int t) { return t == GGUF_F32 || t == GGUF_F16 || t == GGUF_BF16; }
static bool is_weight(int t) {
    return t == GGUF_Q8_0 || t == GGUF_Q4_0 || t == GGUF_Q4_K || t == GGUF_Q5_K || t == GGUF_Q6_K ||
           t == GGUF_MXFP4;
}
static int64_t esize(int t) { return t == GGUF_F32 ? 4 : 2; }
static int64_t row_size(int t, int64_t k) {
    const int64_t be = block_elems(t);
    if (be == 0 || k < 0 || k % be) return -1;
    return k / be * block_bytes(t);
}
static size_t align256(size_t v) { return (v + 255) & ~size_t(255); }
static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Which engine runs a dense product of m activation rows of length k: MMVQ
// holds one 32-value piece per thread (k <= 16384); MMQ takes the rest.
// MMQ above mmvq_max_m tokens (and for K > 16384), except Q4_K products that
// the tensor-core MMVQ takes in one launch (up to mmvq_tc_max_m tokens)
static bool use_mmq(int wt, int64_t m, int64_t k) {
    if (k > 16384) return true;
    if (m <= g_mmvq_max_m || g_mmq_enable == 0) return false;
    return !mmvq_tc_wide(wt, k, m);
}

}  // namespace gg

using namespace gg;

extern "C" {

const char *gguf_last_error(void) { return g_last_error.c_str(); }

int64_t gguf_type_block_elems(int type) { return block_elems(type); }
int64_t gguf_type_block_bytes(int type) { return block_bytes(type); }
int64_t gguf_row_size(int type, int64_t k) { return row_size(type, k); }

gguf_status gguf_quantize_q8_1(const void *x, int xt, int64_t m, int64_t k, int64_t ldx, void *xq,
                               gguf_stream_t stream) {
    if (!is_float(xt)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "quantize_q8_1: x type %d is not F32/BF16/F16", xt);
    if (m < 0 || k < 0) return fail(GGUF_ERR_INVALID_ARG, "quantize_q8_1: negative size");
    if (k % 32) return fail(GGUF_ERR_SHAPE, "quantize_q8_1: k=%lld is not a multiple of 32", (long long)k);
    if (ldx < k) return fail(GGUF_ERR_INVALID_ARG, "quantize_q8_1: ldx=%lld < k=%lld", (long long)ldx, (long long)k);
    if (m == 0 || k == 0) return GGUF_OK;
    if (!x || !xq) return fail(GGUF_ERR_INVALID_ARG, "quantize_q8_1: null pointer");
    if (!aligned(x, esize(xt)) || !aligned(xq, 4))
        return fail(GGUF_ERR_ALIGNMENT, "quantize_q8_1: x must be element-aligned and xq 4-byte aligned");
    return cuda_status(launch_quantize_q8_1(x, xt, m, k, ldx, (uint8_t *)xq, nullptr, nullptr, (cudaStream_t)stream),
                       "quantize_q8_1");
}

gguf_status gguf_dequantize(const void *w, int wt, int64_t rows, int64_t k, void *out, int ot, gguf_stream_t stream) {
    if (!is_float(ot)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "dequantize: out type %d is not F32/BF16/F16", ot);
    if (!is_weight(wt) && wt != GGUF_Q8_1 && !is_float(wt))
        return fail(GGUF_ERR_UNSUPPORTED_TYPE, "dequantize: no converter for type %d", wt);
    if (rows < 0 || k < 0) return fail(GGUF_ERR_INVALID_ARG, "dequantize: negative size");
    if (row_size(wt, k) < 0) return fail(GGUF_ERR_SHAPE, "dequantize: k=%lld not a multiple of the block of type %d", (long long)k, wt);
    if (rows == 0 || k == 0) return GGUF_OK;
    if (!w || !out) return fail(GGUF_ERR_INVALID_ARG, "dequantize: null pointer");
    if (is_float(wt)) {
        if (!aligned(w, esize(wt)) || !aligned(out, esize(ot))) return fail(GGUF_ERR_ALIGNMENT, "dequantize: misaligned float buffer");
        if (wt == ot)
            return cuda_status(cudaMemcpyAsync(out, w, (size_t)(rows * k * esize(wt)), cudaMemcpyDeviceToDevice,
                                               (cudaStream_t)stream), "dequantize copy");
        return cuda_status(launch_convert_float(w, wt, rows * k, out, ot, (cudaStream_t)stream), "dequantize convert");
    }
    if (!aligned(w, 16) || !aligned(out, 16)) return fail(GGUF_ERR_ALIGNMENT, "dequantize: w and out must be 16-byte aligned");
    return cuda_status(launch_dequantize((const uint8_t *)w, wt, rows, k, nullptr, rows, out, ot, (cudaStream_t)stream),
                       "dequantize");
}

// whether a kernel may read or write p: device or managed memory, or pinned
// host memory mapped into the unified address space (pageable host memory is
// not accessible, and a kernel touching it would fault)
static bool device_accessible(const void *p) {
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return true;
    return a.type == cudaMemoryTypeHost && a.devicePointer == p;
}

gguf_status gguf_copy_async(void *dst, const void *src, int64_t bytes, gguf_stream_t stream) {
    if (bytes < 0) return fail(GGUF_ERR_INVALID_ARG, "copy_async: negative size");
    if (bytes == 0) return GGUF_OK;
    if (!dst || !src) return fail(GGUF_ERR_INVALID_ARG, "copy_async: null pointer");
    if (!device_accessible(dst) || !device_accessible(src))
        return fail(GGUF_ERR_INVALID_ARG, "copy_async: both buffers must be device, managed or pinned host memory");
    const uintptr_t d = reinterpret_cast<uintptr_t>(dst), s = reinterpret_cast<uintptr_t>(src);
    if (d < s + (uintptr_t)bytes && s < d + (uintptr_t)bytes)
        return fail(GGUF_ERR_INVALID_ARG, "copy_async: the buffers overlap");
    return cuda_status(launch_copy(dst, src, bytes, (cudaStream_t)stream), "copy_async");
}

gguf_status gguf_get_rows(const void *table, int tt, int64_t rows, int64_t k, const int32_t *ids, int64_t n_ids,
                          void *out, int ot, gguf_stream_t stream) {
    if (!is_float(ot)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "get_rows: out type %d is not F32/BF16/F16", ot);
    if (!is_weight(tt) && tt != GGUF_Q8_1) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "get_rows: table type %d not supported", tt);
    if (rows < 0 || k < 0 || n_ids < 0) return fail(GGUF_ERR_INVALID_ARG, "get_rows: negative size");
    if (row_size(tt, k) < 0) return fail(GGUF_ERR_SHAPE, "get_rows: k=%lld not a multiple of the block", (long long)k);
    if (n_ids == 0 || k == 0) return GGUF_OK;
    if (!ids || !out || (rows > 0 && !table)) return fail(GGUF_ERR_INVALID_ARG, "get_rows: null pointer");
    if ((rows > 0 && !aligned(table, 16)) || !aligned(out, 16) || !aligned(ids, 4))
        return fail(GGUF_ERR_ALIGNMENT, "get_rows: table and out must be 16-byte aligned");
    if (rows == 0)  // every id is out of range: all rows are zero
        return cuda_status(cudaMemsetAsync(out, 0, (size_t)(n_ids * k * esize(ot)), (cudaStream_t)stream), "get_rows");
    return cuda_status(launch_dequantize((const uint8_t *)table, tt, n_ids, k, ids, rows, out, ot, (cudaStream_t)stream),
                       "get_rows");
}

size_t gguf_mul_mat_ws_size(int wt, int64_t n, int64_t k, int xt, int64_t m, int yt) {
    if (m <= 0 || k <= 0 || k % 32) return 0;
    if (use_mmq(wt, m, k) && lib_engine(m, k, yt))   // fp16 activation rows, the fp16 weights, fp32 rows (BF16 out)
        return align256((size_t)(m * k * 2)) + align256((size_t)(n * k * 2)) +
               (yt == GGUF_BF16 ? align256((size_t)(m * n * 4)) : 0);
    if (use_mmq(wt, m, k)) {
        // fp16 operand rows (plus their low parts for fp32 outputs), plus fp32
        // partial sums when K is split across CTAs (small m)
        const int64_t kx = op_pitch(wt, k);
        size_t b = align256((size_t)(m * kx * 2));
        if (yt == GGUF_F32) b += align256((size_t)(m * kx * 2));
        if (m <= 256) b += align256((size_t)(m * n * 4));
        return b;
    }
    if (xt == GGUF_Q8_1) return 0;
    return align256((size_t)(m * row_size(GGUF_Q8_1, k)));             // q8_1 rows
}

// The body shared by gguf_mul_mat and gguf_mul_mat_segments: x is quantized
// once for every segment; in the MMVQ range one launch covers all segments.
static gguf_status mul_mat_impl(int wt, const gguf_segment *segs, int nseg, int64_t k, const void *x, int xt,
                                int64_t m, int64_t ldx, int yt, void *ws, size_t ws_bytes, gguf_stream_t stream,
                                const char *what) {
    if (!is_weight(wt)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "%s: weight type %d not supported", what, wt);
    if (!is_float(xt) && xt != GGUF_Q8_1) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "%s: x type %d not supported", what, xt);
    if (!is_float(yt)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "%s: y type %d is not F32/BF16/F16", what, yt);
    if (nseg < 1 || nseg > GGUF_MAX_SEGMENTS || !segs)
        return fail(GGUF_ERR_INVALID_ARG, "%s: %d segments (1..%d)", what, nseg, GGUF_MAX_SEGMENTS);
    if (k < 0 || m < 0) return fail(GGUF_ERR_INVALID_ARG, "%s: negative size", what);
    if (row_size(wt, k) < 0) return fail(GGUF_ERR_SHAPE, "%s: k=%lld not a multiple of the block of type %d", what, (long long)k, wt);
    if (is_float(xt) && ldx < k) return fail(GGUF_ERR_INVALID_ARG, "%s: ldx=%lld < k=%lld", what, (long long)ldx, (long long)k);
    int64_t n_max = 0, n_tot = 0;
    for (int i = 0; i < nseg; i++) {
        const gguf_segment &g = segs[i];
        if (g.n < 0) return fail(GGUF_ERR_INVALID_ARG, "%s: negative size", what);
        if (g.ldy < g.n) return fail(GGUF_ERR_INVALID_ARG, "%s: ldy=%lld < n=%lld", what, (long long)g.ldy, (long long)g.n);
        n_max = g.n > n_max ? g.n : n_max;
        n_tot += g.n;
    }
    if (m == 0 || n_tot == 0) return GGUF_OK;   // nothing to compute: pointers are not looked at
    for (int i = 0; i < nseg; i++) {
        const gguf_segment &g = segs[i];
        if (g.n == 0) continue;
        if (!g.w || !g.y) return fail(GGUF_ERR_INVALID_ARG, "%s: null pointer", what);
        if (!aligned(g.w, 16)) return fail(GGUF_ERR_ALIGNMENT, "%s: weight base must be 16-byte aligned", what);
        if (!aligned(g.y, esize(yt))) return fail(GGUF_ERR_ALIGNMENT, "%s: misaligned y", what);
    }
    if (k == 0) return fail(GGUF_ERR_SHAPE, "%s: k must be positive", what);
    if (!x) return fail(GGUF_ERR_INVALID_ARG, "%s: null pointer", what);
    if ((is_float(xt) && !aligned(x, esize(xt))) || (xt == GGUF_Q8_1 && !aligned(x, 4)))
        return fail(GGUF_ERR_ALIGNMENT, "%s: misaligned x", what);
    const size_t need = gguf_mul_mat_ws_size(wt, n_max, k, xt, m, yt);
    if (ws_bytes < need || (need > 0 && !ws))
        return fail(GGUF_ERR_WORKSPACE, "%s: workspace of %zu bytes < required %zu", what, ws_bytes, need);
    if (need > 0 && !aligned(ws, 16)) return fail(GGUF_ERR_ALIGNMENT, "%s: workspace must be 16-byte aligned", what);
    cudaStream_t s = (cudaStream_t)stream;

    if (use_mmq(wt, m, k) && lib_engine(m, k, yt)) {
        // dequantize + library GEMM: the activations' fp16 operand d16 * q (no
        // min-term correction columns), each weight matrix dequantized to fp16
        uint16_t *xh = (uint16_t *)ws;
        uint16_t *wh = (uint16_t *)((uint8_t *)ws + align256((size_t)(m * k * 2)));
        float *yf = (float *)((uint8_t *)wh + align256((size_t)(n_max * k * 2)));   // BF16 out: fp32 rows first
        cudaError_t e = xt == GGUF_Q8_1 ? launch_q8_1_to_f16((const uint8_t *)x, m, k, xh, nullptr, s, k)
                                        : launch_quantize_q8_1(x, xt, m, k, ldx, nullptr, xh, nullptr, s, k);
        if (e != cudaSuccess) return cuda_status(e, what);
        for (int i = 0; i < nseg; i++) {
            if (segs[i].n == 0) continue;
            if ((e = launch_dequantize((const uint8_t *)segs[i].w, wt, segs[i].n, k, nullptr, 0, wh, GGUF_F16, s)) !=
                cudaSuccess)
                return cuda_status(e, what);
            e = yt == GGUF_BF16 ? library_gemm_f16(wh, xh, segs[i].n, m, k, yf, GGUF_F32, segs[i].n, s)
                                : library_gemm_f16(wh, xh, segs[i].n, m, k, segs[i].y, yt, segs[i].ldy, s);
            if (e == cudaErrorNotSupported)
                return fail(GGUF_ERR_CUDA, "%s: option mmq_engine = 1 needs cuBLAS, which could not be loaded", what);
            if (e == cudaSuccess && yt == GGUF_BF16)
                e = launch_convert_rows(yf, m, segs[i].n, segs[i].y, yt, segs[i].ldy, s);
            if (e != cudaSuccess) return cuda_status(e, what);
        }
        return GGUF_OK;
    }
    if (use_mmq(wt, m, k)) {
        const int64_t kx = op_pitch(wt, k);
        uint8_t *wp = (uint8_t *)ws;
        uint16_t *xh = (uint16_t *)wp;
        wp += align256((size_t)(m * kx * 2));
        uint16_t *xl = nullptr;
        if (yt == GGUF_F32) {
            xl = (uint16_t *)wp;
            wp += align256((size_t)(m * kx * 2));
        }
        float *yacc = (m <= 256 && g_mmq_split_k) ? (float *)wp : nullptr;
        cudaError_t e = xt == GGUF_Q8_1 ? launch_q8_1_to_f16((const uint8_t *)x, m, k, xh, xl, s, kx)
                                        : launch_quantize_q8_1(x, xt, m, k, ldx, nullptr, xh, xl, s, kx);
        if (e != cudaSuccess) return cuda_status(e, what);
        for (int i = 0; i < nseg; i++) {
            if (segs[i].n == 0) continue;
            e = launch_mmq((const uint8_t *)segs[i].w, wt, segs[i].n, k, xh, xl, m, segs[i].y, yt, segs[i].ldy, yacc, s);
            if (e != cudaSuccess) return cuda_status(e, what);
        }
        return GGUF_OK;
    }
    const uint8_t *xq = (const uint8_t *)x;
    if (xt != GGUF_Q8_1) {
        cudaError_t e = launch_quantize_q8_1(x, xt, m, k, ldx, (uint8_t *)ws, nullptr, nullptr, s);
        if (e != cudaSuccess) return cuda_status(e, what);
        xq = (const uint8_t *)ws;
    }
    const int64_t xrb = row_size(GGUF_Q8_1, k);
    const int64_t ysz = esize(yt);
    // MMVQ handles up to 8 rows per launch, or all of them on the wide tensor-core path
    const int64_t chunk = mmvq_tc_wide(wt, k, m) ? m : 8;
    for (int64_t m0 = 0; m0 < m; m0 += chunk) {
        const int64_t mc = m - m0 < chunk ? m - m0 : chunk;
        MmvqSegs sg{};
        for (int i = 0; i < MMVQ_MAX_SEGS; i++) sg.end[i] = INT64_MAX;
        int64_t acc = 0;
        for (int i = 0; i < nseg; i++) {
            if (segs[i].n == 0) continue;
            acc += segs[i].n;
            sg.end[sg.nseg] = acc;
            sg.w[sg.nseg] = (const uint8_t *)segs[i].w;
            sg.y[sg.nseg] = (uint8_t *)segs[i].y + m0 * segs[i].ldy * ysz;
            sg.ldy[sg.nseg] = segs[i].ldy;
            sg.nseg++;
        }
        cudaError_t e = launch_mmvq(sg, wt, k, xq + m0 * xrb, mc, yt, s);
        if (e != cudaSuccess) return cuda_status(e, what);
    }
    return GGUF_OK;
}

gguf_status gguf_mul_mat(const void *w, int wt, int64_t n, int64_t k, const void *x, int xt, int64_t m, int64_t ldx,
                         void *y, int yt, int64_t ldy, void *ws, size_t ws_bytes, gguf_stream_t stream) {
    const gguf_segment seg = {w, n, y, ldy};
    return mul_mat_impl(wt, &seg, 1, k, x, xt, m, ldx, yt, ws, ws_bytes, stream, "mul_mat");
}

size_t gguf_mul_mat_segments_ws_size(int wt, const gguf_segment *segs, int nseg, int64_t k, int xt, int64_t m, int yt) {
    if (!segs || nseg < 1 || nseg > GGUF_MAX_SEGMENTS) return 0;
    int64_t n_max = 0;
    for (int i = 0; i < nseg; i++) n_max = segs[i].n > n_max ? segs[i].n : n_max;
    return gguf_mul_mat_ws_size(wt, n_max, k, xt, m, yt);
}

gguf_status gguf_mul_mat_segments(int wt, const gguf_segment *segs, int nseg, int64_t k, const void *x, int xt,
                                  int64_t m, int64_t ldx, int yt, void *ws, size_t ws_bytes, gguf_stream_t stream) {
    return mul_mat_impl(wt, segs, nseg, k, x, xt, m, ldx, yt, ws, ws_bytes, stream, "mul_mat_segments");
}

// The batch of decode-sized products behind gguf_mul_mat_batch and
// gguf_mul_mat_batch_typed: every job validated before any launch, then one
// chain of programmatic dependent launches closed by an ordinary empty one.
static gguf_status mul_mat_batch_impl(const char *what, const gguf_mm_job_typed *jobs, int njobs, int yt,
                                      gguf_stream_t stream) {
    if (!is_float(yt)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "%s: y type %d is not F32/BF16/F16", what, yt);
    if (njobs < 0 || njobs > GGUF_MAX_BATCH_JOBS || (njobs > 0 && !jobs))
        return fail(GGUF_ERR_INVALID_ARG, "%s: %d jobs (0..%d)", what, njobs, GGUF_MAX_BATCH_JOBS);
    MmvqSegs sgs[GGUF_MAX_BATCH_JOBS];
    int live = 0;
    for (int j = 0; j < njobs; j++) {
        const gguf_mm_job_typed &jb = jobs[j];
        const int wt = jb.wt;
        const int64_t k = jb.k;
        if (!is_weight(wt)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "%s: job %d: weight type %d not supported", what, j, wt);
        if (k < 0) return fail(GGUF_ERR_INVALID_ARG, "%s: job %d: negative size", what, j);
        if (row_size(wt, k) < 0)
            return fail(GGUF_ERR_SHAPE, "%s: job %d: k=%lld not a multiple of the block of type %d", what, j, (long long)k, wt);
        if (jb.nseg < 1 || jb.nseg > GGUF_MAX_SEGMENTS || !jb.segs)
            return fail(GGUF_ERR_INVALID_ARG, "%s: job %d has %d segments (1..%d)", what, j, jb.nseg, GGUF_MAX_SEGMENTS);
        if (jb.m < 0) return fail(GGUF_ERR_INVALID_ARG, "%s: job %d: negative m", what, j);
        MmvqSegs &sg = sgs[j];
        sg = MmvqSegs{};
        for (int i = 0; i < MMVQ_MAX_SEGS; i++) sg.end[i] = INT64_MAX;
        int64_t acc = 0;
        for (int i = 0; i < jb.nseg; i++) {
            const gguf_segment &g = jb.segs[i];
            if (g.n < 0 || g.ldy < g.n) return fail(GGUF_ERR_INVALID_ARG, "%s: job %d segment %d: bad n / ldy", what, j, i);
            if (g.n == 0) continue;
            if (!g.w || !g.y) return fail(GGUF_ERR_INVALID_ARG, "%s: job %d: null pointer", what, j);
            if (!aligned(g.w, 16) || !aligned(g.y, esize(yt)))
                return fail(GGUF_ERR_ALIGNMENT, "%s: job %d: weight base must be 16-byte aligned, y element-aligned", what, j);
            acc += g.n;
            sg.end[sg.nseg] = acc;
            sg.w[sg.nseg] = (const uint8_t *)g.w;
            sg.y[sg.nseg] = g.y;
            sg.ldy[sg.nseg] = g.ldy;
            sg.nseg++;
        }
        if (jb.m == 0 || acc == 0) continue;   // nothing to compute
        if (k == 0) return fail(GGUF_ERR_SHAPE, "%s: job %d: k must be positive", what, j);
        if (!jb.xq || !aligned(jb.xq, 4)) return fail(GGUF_ERR_ALIGNMENT, "%s: job %d: q8_1 input null or misaligned", what, j);
        if (use_mmq(wt, jb.m, k) || (jb.m > 8 && !mmvq_tc_wide(wt, k, jb.m)))
            return fail(GGUF_ERR_INVALID_ARG, "%s: job %d: m=%lld is not decode-sized (the MMVQ range)", what, j,
                        (long long)jb.m);
        live++;
    }
    cudaStream_t s = (cudaStream_t)stream;
    int pos = 0;
    for (int j = 0; j < njobs; j++) {
        MmvqSegs &sg = sgs[j];
        if (jobs[j].m == 0 || sg.nseg == 0) continue;
        sg.chain = live == 1 ? 0 : (pos == 0 ? 1 : 2);
        pos++;
        cudaError_t e = launch_mmvq(sg, jobs[j].wt, jobs[j].k, (const uint8_t *)jobs[j].xq, jobs[j].m, yt, s);
        if (e != cudaSuccess) return cuda_status(e, what);
    }
    if (live > 1) return cuda_status(launch_mmvq_join(s), what);
    return GGUF_OK;
}

gguf_status gguf_mul_mat_batch(int wt, int64_t k, const gguf_mm_job *jobs, int njobs, int yt, gguf_stream_t stream) {
    const char *what = "mul_mat_batch";
    if (!is_weight(wt)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "%s: weight type %d not supported", what, wt);
    if (!is_float(yt)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "%s: y type %d is not F32/BF16/F16", what, yt);
    if (njobs < 0 || njobs > GGUF_MAX_BATCH_JOBS || (njobs > 0 && !jobs))
        return fail(GGUF_ERR_INVALID_ARG, "%s: %d jobs (0..%d)", what, njobs, GGUF_MAX_BATCH_JOBS);
    if (k < 0) return fail(GGUF_ERR_INVALID_ARG, "%s: negative size", what);
    if (row_size(wt, k) < 0) return fail(GGUF_ERR_SHAPE, "%s: k=%lld not a multiple of the block of type %d", what, (long long)k, wt);
    gguf_mm_job_typed tj[GGUF_MAX_BATCH_JOBS];
    for (int j = 0; j < njobs; j++) tj[j] = gguf_mm_job_typed{wt, k, jobs[j].segs, jobs[j].nseg, jobs[j].xq, jobs[j].m};
    return mul_mat_batch_impl(what, tj, njobs, yt, stream);
}

gguf_status gguf_mul_mat_batch_typed(const gguf_mm_job_typed *jobs, int njobs, int yt, gguf_stream_t stream) {
    return mul_mat_batch_impl("mul_mat_batch_typed", jobs, njobs, yt, stream);
}

// ---------------------------------------------------------------- MoE

static gguf_status check_bank(const char *what, const void *w, int wt, int64_t E, int64_t stride, int64_t n, int64_t k) {
    if (!is_weight(wt)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "%s: weight type %d not supported", what, wt);
    if (E <= 0 || n <= 0 || k <= 0) return fail(GGUF_ERR_INVALID_ARG, "%s: experts, n and k must be positive", what);
    if (row_size(wt, k) < 0) return fail(GGUF_ERR_SHAPE, "%s: k=%lld not a multiple of the block of type %d", what, (long long)k, wt);
    if (stride < n * row_size(wt, k)) return fail(GGUF_ERR_INVALID_ARG, "%s: expert stride %lld < n * row_size", what, (long long)stride);
    if (stride % 16) return fail(GGUF_ERR_ALIGNMENT, "%s: expert stride must be a multiple of 16 bytes", what);
    if (!w) return fail(GGUF_ERR_INVALID_ARG, "%s: null weight bank", what);
    if (!aligned(w, 16)) return fail(GGUF_ERR_ALIGNMENT, "%s: weight bank must be 16-byte aligned", what);
    return GGUF_OK;
}

// workspace of one mul_mat_id call
static MoeWs moe_call_layout(const gguf_moe_args *a, void *base) {
    const int64_t R = a->n_tokens * a->top_k;
    const int64_t kx = op_pitch(a->wt, a->k);
    // the grouped GEMMs' fp16 operand holds one row per route, in grouped order
    if (a->mode == GGUF_MOE_GATE_UP_SWIGLU)
        return moe_ws_layout(base, a->n_experts, R, R * kx, 0, 0, false, a->n_tokens <= MOE_VEC_CAP ? a->n : 0);
    return moe_ws_layout(base, a->n_experts, R, R * kx, R * ((a->n + 127) / 128 * 128), 0, false);
}

// The grouped down GEMM with the expert-weighted sum: fp32 atomics into the
// zeroed token rows (the first T * n floats of the z buffer) and one
// conversion to the output dtype; or, with option moe_deterministic, the
// per-route rows z and the slot-order sum.
static cudaError_t grouped_down_sum(const uint8_t *wd, int wt, int64_t stride, int64_t n, int64_t k,
                                    const uint16_t *xh, const uint16_t *xl, int64_t top_k, int64_t T, int64_t E,
                                    const MoeWs &w, const int32_t *ids, const float *route_w, void *y, int yt,
                                    bool precise, cudaStream_t s) {
    const int64_t R = T * top_k;
    cudaError_t e;
    if (g_moe_deterministic) {
        if ((e = launch_moe_down(wd, wt, stride, n, k, xh, xl, top_k, R, E, w, w.z, precise, s)) != cudaSuccess)
            return e;
        return launch_moe_finalize(w.z, w.pos, ids, w.offsets, route_w, T, top_k, n, y, yt, s);
    }
    if ((e = cudaMemsetAsync(w.z, 0, sizeof(float) * (size_t)(T * n), s)) != cudaSuccess) return e;
    if ((e = launch_moe_down(wd, wt, stride, n, k, xh, xl, top_k, R, E, w, w.z, precise, s, w.z, route_w)) !=
        cudaSuccess)
        return e;
    return launch_convert_rows(w.z, T, n, y, yt, n, s);
}

// the route-batched MMVQ path: few tokens, and weight rows it takes
static bool moe_vec(int64_t n_tokens, int wt, int64_t k) {
    return n_tokens <= g_moe_vec_max_tokens && mmvq_routes_supported(wt, k);
}

static gguf_status check_moe(const gguf_moe_args *a) {
    if (!a) return fail(GGUF_ERR_INVALID_ARG, "mul_mat_id: null args");
    gguf_status st = check_bank("mul_mat_id", a->w, a->wt, a->n_experts, a->expert_stride, a->n, a->k);
    if (st != GGUF_OK) return st;
    if (a->n_tokens < 0 || a->top_k <= 0) return fail(GGUF_ERR_INVALID_ARG, "mul_mat_id: bad n_tokens / top_k");
    if (a->n_tokens * a->top_k > INT32_MAX) return fail(GGUF_ERR_INVALID_ARG, "mul_mat_id: too many routes");
    if (!is_float(a->xt) && a->xt != GGUF_Q8_1) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "mul_mat_id: x type %d", a->xt);
    if (is_float(a->xt) && a->ldx < a->k) return fail(GGUF_ERR_INVALID_ARG, "mul_mat_id: ldx < k");
    if (a->k % 8) return fail(GGUF_ERR_SHAPE, "mul_mat_id: k must be a multiple of 8");
    if (a->mode == GGUF_MOE_GATE_UP_SWIGLU) {
        if (a->n % 128) return fail(GGUF_ERR_SHAPE, "mul_mat_id gate_up: n = 2*I must be a multiple of 128");
        if (a->yt != GGUF_BF16 && a->yt != GGUF_Q8_1 && a->yt != GGUF_F16)
            return fail(GGUF_ERR_UNSUPPORTED_TYPE, "mul_mat_id gate_up: out type %d is not BF16/Q8_1/F16", a->yt);
    } else if (a->mode == GGUF_MOE_DOWN_WEIGHTED_SUM || a->mode == GGUF_MOE_PLAIN) {
        if (!is_float(a->yt)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "mul_mat_id: out type %d", a->yt);
    } else {
        return fail(GGUF_ERR_INVALID_ARG, "mul_mat_id: unknown mode %d", a->mode);
    }
    if (a->n_tokens > 0 && (!a->x || !a->ids || !a->y)) return fail(GGUF_ERR_INVALID_ARG, "mul_mat_id: null pointer");
    if (a->n_tokens > 0 && (!aligned(a->ids, 4) || !aligned(a->x, a->xt == GGUF_Q8_1 ? 4 : esize(a->xt)) ||
                            !aligned(a->y, a->yt == GGUF_F32 ? 4 : 2)))
        return fail(GGUF_ERR_ALIGNMENT, "mul_mat_id: misaligned x, ids or y");
    return GGUF_OK;
}

// the fp16 operand of the grouped GEMMs in grouped route order: x row i
// feeds the routes i * fan + j, j < fan (fan = top_k: token rows; 1: route
// rows), each written at its expert offset + slot
static cudaError_t to_f16_operand(const void *x, int xt, int64_t R, int64_t k, int64_t ldx, uint16_t *xh,
                                  uint16_t *xl, int64_t pitch, const MoeWs &w, const int32_t *ids, int32_t fan,
                                  cudaStream_t s) {
    const int64_t rows = R / fan;
    return xt == GGUF_Q8_1
               ? launch_q8_1_to_f16((const uint8_t *)x, rows, k, xh, xl, s, pitch, ids, w.pos, w.offsets, fan)
               : launch_quantize_q8_1(x, xt, rows, k, ldx, nullptr, xh, xl, s, pitch, ids, w.pos, w.offsets, fan);
}

size_t gguf_mul_mat_id_ws_size(const gguf_moe_args *args) {
    if (!args || args->n_experts <= 0 || args->top_k <= 0 || args->n_tokens < 0) return 0;
    return moe_call_layout(args, nullptr).bytes;
}

gguf_status gguf_mul_mat_id(const gguf_moe_args *a, void *ws, size_t ws_bytes, gguf_stream_t stream) {
    gguf_status st = check_moe(a);
    if (st != GGUF_OK) return st;
    if (a->n_tokens == 0) return GGUF_OK;
    const size_t need = moe_call_layout(a, nullptr).bytes;
    if (!ws || ws_bytes < need) return fail(GGUF_ERR_WORKSPACE, "mul_mat_id: workspace of %zu bytes < required %zu", ws_bytes, need);
    if (!aligned(ws, 256)) return fail(GGUF_ERR_ALIGNMENT, "mul_mat_id: workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    const MoeWs w = moe_call_layout(a, ws);
    const int64_t R = a->n_tokens * a->top_k;
    const int bn = moe_bn(R, a->n_experts);
    cudaError_t e;
    const bool vec = moe_vec(a->n_tokens, a->wt, a->k);
    const bool plain = a->mode == GGUF_MOE_PLAIN;
    if (vec) {
        // route-batched MMVQ: each active route reads its expert's rows once
        const int64_t rows = a->mode == GGUF_MOE_DOWN_WEIGHTED_SUM ? R : a->n_tokens;
        const bool gu = a->mode == GGUF_MOE_GATE_UP_SWIGLU;
        const bool weighted = a->mode == GGUF_MOE_DOWN_WEIGHTED_SUM;
        // the route marks ride on the quantize launch when there is one
        const uint8_t *xq = (const uint8_t *)a->x;
        if (a->xt != GGUF_Q8_1) {
            RouteMarks mk;
            mk.ids = a->ids;
            mk.rw = weighted ? a->route_w : nullptr;
            mk.R = R;
            mk.E = a->n_experts;
            mk.skip_zero_w = weighted ? 1 : 0;
            mk.pos = w.pos;
            mk.status = a->dev_status;
            if ((e = launch_quantize_q8_1(a->x, a->xt, rows, a->k, a->ldx, (uint8_t *)w.xh, nullptr, nullptr, s, 0,
                                          nullptr, nullptr, nullptr, 1, mk)) != cudaSuccess)
                return cuda_status(e, "mul_mat_id quantize");
            xq = (const uint8_t *)w.xh;
        } else if ((e = moe_mark(a->ids, weighted ? a->route_w : nullptr, R, a->n_experts, weighted, a->dev_status,
                                 w.pos, s)) != cudaSuccess) {
            return cuda_status(e, "mul_mat_id routes");
        }
        const MmvqRoutes rt{a->ids, w.pos, a->expert_stride, a->top_k, weighted ? 1 : 0};
        if (plain) {
            if ((e = launch_mmvq_routes(a->wt, (const uint8_t *)a->w, rt, a->n, a->k, xq, R, w.z, s)) != cudaSuccess)
                return cuda_status(e, "mul_mat_id");
            return cuda_status(launch_moe_plain_store(w.z, w.pos, nullptr, nullptr, R, a->n, a->y, a->yt, s),
                               "mul_mat_id store");
        }
        if (!gu) {
            if ((e = launch_mmvq_routes(a->wt, (const uint8_t *)a->w, rt, a->n, a->k, xq, R, w.z, s)) != cudaSuccess)
                return cuda_status(e, "mul_mat_id down");
            return cuda_status(launch_moe_finalize(w.z, w.pos, nullptr, nullptr, a->route_w, a->n_tokens, a->top_k, a->n,
                                                   a->y, a->yt, s),
                               "mul_mat_id finalize");
        }
        const int64_t idim = a->n / 2;
        if ((e = launch_mmvq_routes(a->wt, (const uint8_t *)a->w, rt, a->n, a->k, xq, R, w.zv, s)) != cudaSuccess)
            return cuda_status(e, "mul_mat_id gate_up");
        uint16_t *h = a->yt == GGUF_BF16 ? (uint16_t *)a->y : w.hb;
        if ((e = launch_moe_swiglu(w.zv, w.pos, R, idim, h, s)) != cudaSuccess) return cuda_status(e, "mul_mat_id swiglu");
        if (a->yt == GGUF_Q8_1)
            e = launch_quantize_q8_1(h, GGUF_BF16, R, idim, idim, (uint8_t *)a->y, nullptr, nullptr, s);
        else if (a->yt == GGUF_F16 && (e = launch_quantize_q8_1(h, GGUF_BF16, R, idim, idim, w.hqv, nullptr, nullptr, s)) == cudaSuccess)
            e = launch_q8_1_to_f16(w.hqv, R, idim, (uint16_t *)a->y, nullptr, s, idim);
        return cuda_status(e, "mul_mat_id gate_up output");
    }
    if (a->mode == GGUF_MOE_GATE_UP_SWIGLU) {
        const int64_t idim = a->n / 2;
        const size_t ybytes = a->yt == GGUF_Q8_1 ? (size_t)(R * row_size(GGUF_Q8_1, idim)) : (size_t)(R * idim * 2);
        if ((e = cudaMemsetAsync(a->y, 0, ybytes, s)) != cudaSuccess) return cuda_status(e, "mul_mat_id");
        if ((e = moe_group(a->ids, nullptr, R, a->n_experts, false, a->dev_status, w, bn, s)) != cudaSuccess) return cuda_status(e, "mul_mat_id grouping");
        uint16_t *xl = g_moe_gate_up_precise ? w.xl : nullptr;
        if ((e = to_f16_operand(a->x, a->xt, R, a->k, a->ldx, w.xh, xl, op_pitch(a->wt, a->k), w, a->ids,
                                (int32_t)a->top_k, s)) != cudaSuccess)
            return cuda_status(e, "mul_mat_id quantize");
        e = launch_moe_gate_up((const uint8_t *)a->w, a->wt, a->expert_stride, a->n, a->k, w.xh, xl, a->top_k, R,
                               a->n_experts, w, a->yt == GGUF_Q8_1 ? (uint8_t *)a->y : nullptr,
                               a->yt == GGUF_BF16 ? (uint16_t *)a->y : nullptr,
                               a->yt == GGUF_F16 ? (uint16_t *)a->y : nullptr, nullptr, a->n / 2, false, s);
        return cuda_status(e, "mul_mat_id gate_up");
    }
    if (plain) {   // token rows, one output row per route
        if ((e = moe_group(a->ids, nullptr, R, a->n_experts, false, a->dev_status, w, bn, s)) != cudaSuccess)
            return cuda_status(e, "mul_mat_id grouping");
        if ((e = to_f16_operand(a->x, a->xt, R, a->k, a->ldx, w.xh, w.xl, op_pitch(a->wt, a->k), w, a->ids,
                                (int32_t)a->top_k, s)) != cudaSuccess)
            return cuda_status(e, "mul_mat_id quantize");
        if ((e = launch_moe_down((const uint8_t *)a->w, a->wt, a->expert_stride, a->n, a->k, w.xh, w.xl, a->top_k, R,
                                 a->n_experts, w, w.z, a->yt == GGUF_F32, s)) != cudaSuccess)
            return cuda_status(e, "mul_mat_id");
        return cuda_status(launch_moe_plain_store(w.z, w.pos, a->ids, w.offsets, R, a->n, a->y, a->yt, s),
                           "mul_mat_id store");
    }
    if ((e = moe_group(a->ids, a->route_w, R, a->n_experts, true, a->dev_status, w, bn, s)) != cudaSuccess) return cuda_status(e, "mul_mat_id grouping");
    if ((e = to_f16_operand(a->x, a->xt, R, a->k, a->ldx, w.xh, w.xl, op_pitch(a->wt, a->k), w, a->ids, 1, s)) !=
        cudaSuccess)
        return cuda_status(e, "mul_mat_id quantize");
    return cuda_status(grouped_down_sum((const uint8_t *)a->w, a->wt, a->expert_stride, a->n, a->k, w.xh, w.xl,
                                        a->top_k, a->n_tokens, a->n_experts, w, a->ids, a->route_w, a->y, a->yt,
                                        a->yt == GGUF_F32, s),
                       "mul_mat_id down");
}

static MoeWs ffn_layout(const gguf_moe_ffn_args *a, void *base) {
    const int64_t R = a->n_tokens * a->top_k;
    return moe_ws_layout(base, a->n_experts, R, R * op_pitch(a->gate_up_type, a->hidden),
                         R * ((a->hidden + 127) / 128 * 128), R * op_pitch(a->down_type, a->inter),
                         a->yt == GGUF_F32 || g_moe_down_precise,
                         a->n_tokens <= MOE_VEC_CAP ? 2 * a->inter : 0);
}

size_t gguf_moe_ffn_ws_size(const gguf_moe_ffn_args *a) {
    if (!a || a->n_experts <= 0 || a->top_k <= 0 || a->n_tokens < 0) return 0;
    return ffn_layout(a, nullptr).bytes;
}

gguf_status gguf_moe_ffn(const gguf_moe_ffn_args *a, void *ws, size_t ws_bytes, gguf_stream_t stream) {
    if (!a) return fail(GGUF_ERR_INVALID_ARG, "moe_ffn: null args");
    gguf_status st = check_bank("moe_ffn gate_up", a->w_gate_up, a->gate_up_type, a->n_experts, a->gate_up_stride,
                                2 * a->inter, a->hidden);
    if (st != GGUF_OK) return st;
    st = check_bank("moe_ffn down", a->w_down, a->down_type, a->n_experts, a->down_stride, a->hidden, a->inter);
    if (st != GGUF_OK) return st;
    if (a->inter % 64) return fail(GGUF_ERR_SHAPE, "moe_ffn: intermediate size must be a multiple of 64");
    if (a->hidden % 8) return fail(GGUF_ERR_SHAPE, "moe_ffn: hidden size must be a multiple of 8");
    if (a->n_tokens < 0 || a->top_k <= 0 || a->n_tokens * a->top_k > INT32_MAX) return fail(GGUF_ERR_INVALID_ARG, "moe_ffn: bad n_tokens / top_k");
    if (!is_float(a->xt) && a->xt != GGUF_Q8_1) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "moe_ffn: x type %d", a->xt);
    if (!is_float(a->yt)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "moe_ffn: y type %d", a->yt);
    if (is_float(a->xt) && a->ldx < a->hidden) return fail(GGUF_ERR_INVALID_ARG, "moe_ffn: ldx < hidden");
    if (a->n_tokens == 0) return GGUF_OK;
    if (!a->x || !a->ids || !a->y) return fail(GGUF_ERR_INVALID_ARG, "moe_ffn: null pointer");
    const size_t need = ffn_layout(a, nullptr).bytes;
    if (!ws || ws_bytes < need) return fail(GGUF_ERR_WORKSPACE, "moe_ffn: workspace of %zu bytes < required %zu", ws_bytes, need);
    if (!aligned(ws, 256)) return fail(GGUF_ERR_ALIGNMENT, "moe_ffn: workspace must be 256-byte aligned");
    cudaStream_t s = (cudaStream_t)stream;
    const MoeWs w = ffn_layout(a, ws);
    const int64_t R = a->n_tokens * a->top_k;
    const int bn = moe_bn(R, a->n_experts);
    cudaError_t e;
    if (moe_vec(a->n_tokens, a->gate_up_type, a->hidden) && mmvq_routes_supported(a->down_type, a->inter)) {
        // route-batched MMVQ for both products: x -> q8_1, gate_up rows per
        // route, SwiGLU -> bf16 -> q8_1, down rows per route, weighted sum
        // the route marks ride on the quantize launch (one launch fewer)
        const uint8_t *xq = (const uint8_t *)a->x;
        if (a->xt != GGUF_Q8_1) {
            RouteMarks mk;
            mk.ids = a->ids;
            mk.rw = a->route_w;
            mk.R = R;
            mk.E = a->n_experts;
            mk.skip_zero_w = 1;
            mk.pos = w.pos;
            mk.status = a->dev_status;
            if ((e = launch_quantize_q8_1(a->x, a->xt, a->n_tokens, a->hidden, a->ldx, (uint8_t *)w.xh, nullptr,
                                          nullptr, s, 0, nullptr, nullptr, nullptr, 1, mk)) != cudaSuccess)
                return cuda_status(e, "moe_ffn quantize");
            xq = (const uint8_t *)w.xh;
        } else if ((e = moe_mark(a->ids, a->route_w, R, a->n_experts, true, a->dev_status, w.pos, s)) != cudaSuccess) {
            return cuda_status(e, "moe_ffn routes");
        }
        uint8_t *hq = (uint8_t *)w.h16;   // q8_1 rows of h ([R][I / 32] blocks fit in the fp16 operand buffer)
        if ((e = launch_mmvq_routes(a->gate_up_type, (const uint8_t *)a->w_gate_up,
                                    MmvqRoutes{a->ids, w.pos, a->gate_up_stride, a->top_k, 0}, 2 * a->inter, a->hidden,
                                    xq, R, w.zv, s)) != cudaSuccess ||
            (e = launch_moe_swiglu_q8_1(w.zv, w.pos, R, a->inter, hq, s)) != cudaSuccess)
            return cuda_status(e, "moe_ffn gate_up");
        if ((e = launch_mmvq_routes(a->down_type, (const uint8_t *)a->w_down,
                                    MmvqRoutes{a->ids, w.pos, a->down_stride, a->top_k, 1}, a->hidden, a->inter, hq, R,
                                    w.z, s)) != cudaSuccess)
            return cuda_status(e, "moe_ffn down");
        return cuda_status(launch_moe_finalize(w.z, w.pos, nullptr, nullptr, a->route_w, a->n_tokens, a->top_k,
                                               a->hidden, a->y, a->yt, s),
                           "moe_ffn finalize");
    }
    // one grouping serves both GEMMs; a route of weight 0 contributes nothing and is skipped by both
    if ((e = moe_group(a->ids, a->route_w, R, a->n_experts, true, a->dev_status, w, bn, s)) != cudaSuccess) return cuda_status(e, "moe_ffn grouping");
    uint16_t *xl = g_moe_gate_up_precise ? w.xl : nullptr;
    if ((e = to_f16_operand(a->x, a->xt, R, a->hidden, a->ldx, w.xh, xl, op_pitch(a->gate_up_type, a->hidden), w,
                            a->ids, (int32_t)a->top_k, s)) != cudaSuccess)
        return cuda_status(e, "moe_ffn quantize");
    if ((e = launch_moe_gate_up((const uint8_t *)a->w_gate_up, a->gate_up_type, a->gate_up_stride, 2 * a->inter,
                                a->hidden, w.xh, xl, a->top_k, R, a->n_experts, w, nullptr, nullptr, w.h16, w.h16lo,
                                op_pitch(a->down_type, a->inter), true, s)) != cudaSuccess)
        return cuda_status(e, "moe_ffn gate_up");
    return cuda_status(grouped_down_sum((const uint8_t *)a->w_down, a->down_type, a->down_stride, a->hidden, a->inter,
                                        w.h16, w.h16lo, a->top_k, a->n_tokens, a->n_experts, w, a->ids, a->route_w,
                                        a->y, a->yt, a->yt == GGUF_F32 || g_moe_down_precise, s),
                       "moe_ffn down");
}

gguf_status gguf_debug_block_dots(const void *w, int wt, int64_t n, int64_t k, const void *xq, int64_t m,
                                  int32_t *sums, gguf_stream_t stream) {
    if (!is_weight(wt)) return fail(GGUF_ERR_UNSUPPORTED_TYPE, "debug_block_dots: weight type %d not supported", wt);
    if (n < 0 || k < 0 || m < 0) return fail(GGUF_ERR_INVALID_ARG, "debug_block_dots: negative size");
    if (row_size(wt, k) < 0) return fail(GGUF_ERR_SHAPE, "debug_block_dots: k not a multiple of the block");
    if (n == 0 || m == 0 || k == 0) return GGUF_OK;
    if (!w || !xq || !sums) return fail(GGUF_ERR_INVALID_ARG, "debug_block_dots: null pointer");
    return cuda_status(launch_block_dots((const uint8_t *)w, wt, n, k, (const uint8_t *)xq, m, sums, (cudaStream_t)stream),
                       "debug_block_dots");
}

gguf_status gguf_set_option(const char *key, int64_t value) {
    if (!key) return fail(GGUF_ERR_INVALID_ARG, "set_option: null key");
    if (!strcmp(key, "mmvq_max_m")) {
        if (value < 0) return fail(GGUF_ERR_INVALID_ARG, "set_option: mmvq_max_m must be >= 0");
        g_mmvq_max_m = value;
        return GGUF_OK;
    }
    if (!strcmp(key, "mmvq_tc")) {
        g_mmvq_tc = value != 0;
        return GGUF_OK;
    }
    if (!strcmp(key, "moe_vec_max_tokens")) {
        if (value < 0 || value > MOE_VEC_CAP) return fail(GGUF_ERR_INVALID_ARG, "set_option: moe_vec_max_tokens must be in [0, 256]");
        g_moe_vec_max_tokens = value;
        return GGUF_OK;
    }
    if (!strcmp(key, "mmvq_tc_min_m")) {
        if (value < 1 || value > 8) return fail(GGUF_ERR_INVALID_ARG, "set_option: mmvq_tc_min_m must be in [1, 8]");
        g_mmvq_tc_min_m = value;
        return GGUF_OK;
    }
    if (!strcmp(key, "mmvq_tc_max_m")) {
        if (value < 8 || value > 32) return fail(GGUF_ERR_INVALID_ARG, "set_option: mmvq_tc_max_m must be in [8, 32]");
        g_mmvq_tc_max_m = value;
        return GGUF_OK;
    }
    if (!strcmp(key, "mmq_enable")) {
        g_mmq_enable = value != 0;
        return GGUF_OK;
    }
    if (!strcmp(key, "mmq_stage")) {
        g_mmq_stage = value != 0;
        return GGUF_OK;
    }
    if (!strcmp(key, "moe_deterministic")) {
        g_moe_deterministic = value != 0;
        return GGUF_OK;
    }
    if (!strcmp(key, "mmq_bn_max")) {
        if (value != 128 && value != 256) return fail(GGUF_ERR_INVALID_ARG, "set_option: mmq_bn_max must be 128 or 256");
        g_mmq_bn_max = value;
        return GGUF_OK;
    }
    if (!strcmp(key, "mmq_split_k")) {
        g_mmq_split_k = value != 0;
        return GGUF_OK;
    }
    if (!strcmp(key, "moe_down_precise")) {
        g_moe_down_precise = value != 0;
        return GGUF_OK;
    }
    if (!strcmp(key, "moe_gate_up_precise")) {
        g_moe_gate_up_precise = value != 0;
        return GGUF_OK;
    }
    if (!strcmp(key, "mmq_engine")) {
        if (value != 0 && value != 1) return fail(GGUF_ERR_INVALID_ARG, "set_option: mmq_engine must be 0 or 1");
        g_mmq_engine = value;
        return GGUF_OK;
    }
    return fail(GGUF_ERR_INVALID_ARG, "set_option: unknown key '%s'", key);
}

int64_t gguf_get_option(const char *key) {
    if (!key) return -1;
    if (!strcmp(key, "mmvq_max_m")) return g_mmvq_max_m;
    if (!strcmp(key, "mmq_enable")) return g_mmq_enable;
    if (!strcmp(key, "mmvq_tc")) return g_mmvq_tc;
    if (!strcmp(key, "mmvq_tc_min_m")) return g_mmvq_tc_min_m;
    if (!strcmp(key, "moe_vec_max_tokens")) return g_moe_vec_max_tokens;
    if (!strcmp(key, "mmvq_tc_max_m")) return g_mmvq_tc_max_m;
    if (!strcmp(key, "mmq_stage")) return g_mmq_stage;
    if (!strcmp(key, "moe_deterministic")) return g_moe_deterministic;
    if (!strcmp(key, "moe_down_precise")) return g_moe_down_precise;
    if (!strcmp(key, "moe_gate_up_precise")) return g_moe_gate_up_precise;
    if (!strcmp(key, "mmq_engine")) return g_mmq_engine;
    if (!strcmp(key, "mmq_bn_max")) return g_mmq_bn_max;
    if (!strcmp(key, "mmq_split_k")) return g_mmq_split_k;
    return -1;
}

}  // extern "C"

