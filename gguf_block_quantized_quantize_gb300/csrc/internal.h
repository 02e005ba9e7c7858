// Host-side launch interface between the C-ABI layer (abi.cu) and the kernel
// translation units.  Every launcher returns the cudaError_t of its launch and
// assumes its arguments were validated by abi.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/gguf_gb300.h"

namespace gg {

struct DeviceInfo {
    int sm_count;
    int cc_major, cc_minor;
    size_t smem_optin;
};
const DeviceInfo &device_info();
// Resident CTAs per SM of kernel `kern` at `threads` per CTA and `smem` bytes
// of dynamic shared memory on the current device (at least 1).  Queried once
// per (device, kernel, threads, smem) and cached, so a launch costs no driver
// query after the first; the kernel's dynamic shared-memory limit is raised
// to the largest smem asked for.  0 with the CUDA error in *err on failure.
int kernel_occupancy(const void *kern, int threads, size_t smem, cudaError_t *err);
// sets the thread-local message returned by gguf_last_error() and returns st
gguf_status report(gguf_status st, const char *msg);

// dst[0, bytes) = src[0, bytes) on the SMs, as a programmatic dependent launch;
// both pointers device-accessible (copy.cu)
cudaError_t launch_copy(void *dst, const void *src, int64_t bytes, cudaStream_t s);

// q8_1 quantization (xq may be null); also writes the fp16 tensor-core operand
// xh[m][pitch] = fp16(d16*q) when xh != nullptr, and its low part
// xl = fp16(d16*q - xh) when xl != nullptr.  pitch > k appends the Q4_K
// / Q5_K min-term correction columns (see op_pitch) and zero padding.
// ids (optional, device; with the MoE grouping's pos and offsets): the fp16
// operand is written in grouped route order, input row i feeding the routes
// r = i * fan + j (j < fan); an active route (pos[r] >= 0) goes to operand
// row offsets[ids[r]] + pos[r], a skipped one nowhere.  Each input row is
// quantized once.
// The route marks of the MoE vector path, written by the same launch when
// ids != nullptr: pos[r] = r for an active route, -1 for one whose expert id
// is outside [0, E) or (skip_zero_w) whose weight is 0; every id >= E adds 1
// to *status (when not null).  The quantization does not wait for them.
struct RouteMarks {
    const int32_t *ids = nullptr;
    const float *rw = nullptr;
    int64_t R = 0, E = 0;
    int skip_zero_w = 0;
    int32_t *pos = nullptr, *status = nullptr;
};
cudaError_t launch_quantize_q8_1(const void *x, int xt, int64_t m, int64_t k, int64_t ldx, uint8_t *xq,
                                 uint16_t *xh, uint16_t *xl, cudaStream_t s, int64_t pitch = 0,
                                 const int32_t *ids = nullptr, const int32_t *pos = nullptr,
                                 const int32_t *offsets = nullptr, int32_t fan = 1, const RouteMarks &marks = {});
// the same fp16 operand(s) from q8_1 rows
cudaError_t launch_q8_1_to_f16(const uint8_t *xq, int64_t m, int64_t k, uint16_t *xh, uint16_t *xl, cudaStream_t s,
                               int64_t pitch = 0, const int32_t *ids = nullptr, const int32_t *pos = nullptr,
                               const int32_t *offsets = nullptr, int32_t fan = 1);
// Row length of the tensor-core operand for weight type wt: k, plus for the
// affine K-quants (Q4_K, Q5_K) one min-term correction column per 32-block,
// rounded up to the 64-value K step.
inline int64_t op_pitch(int wt, int64_t k) {
    return (wt == GGUF_Q4_K || wt == GGUF_Q5_K) ? (k + k / 32 + 63) / 64 * 64 : k;
}

cudaError_t launch_dequantize(const uint8_t *w, int wt, int64_t rows, int64_t k, const int32_t *ids,
                              int64_t table_rows, void *out, int ot, cudaStream_t s);
cudaError_t launch_convert_float(const void *x, int xt, int64_t count, void *out, int ot, cudaStream_t s);
cudaError_t launch_block_dots(const uint8_t *w, int wt, int64_t n, int64_t k, const uint8_t *xq, int64_t m,
                              int32_t *sums, cudaStream_t s);

// option "mmvq_tc": 5..8 tokens of Q4_K rows run on the tensor-core MMVQ (1, default) or dp4a (0)
int64_t option_mmvq_tc();
int64_t option_mmvq_tc_min_m();
// option "mmvq_tc_max_m" (default 32): Q4_K products of 9..this many tokens run
// as one tensor-core MMVQ launch instead of MMQ
int64_t option_mmvq_tc_max_m();
// option "mmq_stage" (default 1): the tensor-core GEMM stages packed weight
// rows in shared memory with bulk tensor copies where their layout allows
int64_t option_mmq_stage();
// option "mmq_bn_max" (128 or 256, default 256): widest activation tile of the
// dense MMQ; tiles of at most 128 rows keep the weight operand in TMEM
int64_t option_mmq_bn_max();
// whether m (> 8) tokens of K-long Q4_K rows take the tensor-core MMVQ
bool mmvq_tc_wide(int wt, int64_t k, int64_t m);

// Weight segments that read the same activations; one MMVQ launch covers all
// of them.  Row r of the launch is row r - end[s-1] of segment s (end[-1] = 0);
// end[] is cumulative and padded with INT64_MAX past nseg.
constexpr int MMVQ_MAX_SEGS = 8;
struct MmvqSegs {
    int nseg;
    int64_t end[MMVQ_MAX_SEGS];
    const uint8_t *w[MMVQ_MAX_SEGS];
    void *y[MMVQ_MAX_SEGS];
    int64_t ldy[MMVQ_MAX_SEGS];
    // programmatic dependent launch: 0 a launch on its own; 1 the first launch
    // of a batch whose launches share inputs written before the batch; 2 a
    // later launch of such a batch (see mmvq_pdl_enter)
    int chain;
    __host__ __device__ int64_t rows() const { return end[nseg - 1]; }
};
// one segment: W[n][k] -> y[.][ldy]
MmvqSegs mmvq_one_segment(const void *w, int64_t n, void *y, int64_t ldy);

// MoE routes of the route-batched MMVQ: grid row blockIdx.y is route slot r
struct MmvqRoutes {
    const int32_t *ids;      // expert of each route slot
    const int32_t *pos;      // < 0: the route is skipped (inactive, out-of-range id or weight 0)
    int64_t expert_stride;   // bytes between the experts' matrices
    int64_t top_k;           // route slots per token
    int x_per_route;         // activation row of route r: r (1) or its token r / top_k (0)
    int pack;                // > 1: one-warp CTAs treat this many consecutive rows as one (set by the launcher)
};
// z[r][n] (fp32) = W[ids[r]] . q8_1 activation row of route r, for every route
// slot r < routes with pos[r] >= 0 (W: the expert bank, [n][k] of type wt per
// expert); one launch, one token per route
cudaError_t launch_mmvq_routes(int wt, const uint8_t *bank, const MmvqRoutes &rt, int64_t n, int64_t k,
                               const uint8_t *xq, int64_t routes, float *z, cudaStream_t s);
// whether launch_mmvq_routes takes rows of k values of type wt
bool mmvq_routes_supported(int wt, int64_t k);

// for every segment s: y_s[m][ldy_s] (yt) = W_s (wt) . q8_1 rows xq[m] ; m <= 8,
// or m <= 32 when mmvq_tc_wide(wt, k, m)
cudaError_t launch_mmvq(const MmvqSegs &sg, int wt, int64_t k, const uint8_t *xq, int64_t m, int yt, cudaStream_t s);
// an empty kernel launched without programmatic serialization: the end of a
// batch of chained launches (sg.chain 1, 2, ...)
cudaError_t launch_mmvq_join(cudaStream_t s);

// tensor-core MMQ: y[m][ldy] = W[n][k] . xh[m][k] (fp16 operand rows; fp32
// outputs also need the low parts xl).  yacc (optional, fp32 [m][n]) lets small
// m split K across CTAs.
cudaError_t launch_mmq(const uint8_t *w, int wt, int64_t n, int64_t k, const uint16_t *xh, const uint16_t *xl,
                       int64_t m, void *y, int yt, int64_t ldy, float *yacc, cudaStream_t s);
cudaError_t launch_convert_rows(const float *yacc, int64_t m, int64_t n, void *y, int yt, int64_t ldy, cudaStream_t s);
// the library-GEMM engine (libgemm.cu): y[m][ldy] (F32 / F16) = X[m][k] .
// W[n][k]^T with fp16 operands and fp32 accumulation, by cuBLAS opened at run
// time; cudaErrorNotSupported when cuBLAS cannot be loaded
cudaError_t library_gemm_f16(const uint16_t *w, const uint16_t *x, int64_t n, int64_t m, int64_t k, void *y, int yt,
                             int64_t ldy, cudaStream_t s);
// option "mmq_engine" (default 0): 1 runs the prefill products with 16-bit
// outputs as dequantize + library GEMM instead of the fused tensor-core MMQ
int64_t option_mmq_engine();

// ---- MoE (moe.cu)
struct MoeWs {
    int32_t *counts, *offsets, *pos, *route_list, *tile_expert, *tile_start, *n_tiles;
    uint16_t *xh, *xl;
    float *z;  // per-route outputs of the down GEMM [R][n]
    uint16_t *h16, *h16lo;
    // route-batched (vector) gate_up: per-route g | u rows [R][2I], h [R][I] bf16, h as q8_1
    float *zv;
    uint16_t *hb;
    uint8_t *hqv;
    size_t bytes;
};
// base == nullptr computes only the size; vec_n2 = 2I reserves the vector
// gate_up buffers (0: none)
MoeWs moe_ws_layout(void *base, int64_t E, int64_t R, int64_t xh_elems, int64_t z_elems, int64_t h16_elems,
                    bool with_lo, int64_t vec_n2 = 0);
// h[r][j] = bf16(silu(g) * u) of the vector gate_up rows z[r] = (g[0..I), u[0..I));
// zeros for skipped routes (pos[r] < 0)
cudaError_t launch_moe_swiglu(const float *z, const int32_t *pos, int64_t R, int64_t I, uint16_t *h, cudaStream_t s);
// the same h quantized to q8_1 rows hq[R][I / 32] in the same pass (the bits
// that launch_moe_swiglu followed by the q8_1 quantize give)
cudaError_t launch_moe_swiglu_q8_1(const float *z, const int32_t *pos, int64_t R, int64_t I, uint8_t *hq,
                                  cudaStream_t s);
int moe_bn(int64_t routes, int64_t experts);
cudaError_t moe_group(const int32_t *ids, const float *rw, int64_t R, int64_t E, bool skip_zero_w, int32_t *status,
                      const MoeWs &w, int bn, cudaStream_t s);
// route marks only (pos[r] = r or -1), for the route-batched path
cudaError_t moe_mark(const int32_t *ids, const float *rw, int64_t R, int64_t E, bool skip_zero_w, int32_t *status,
                     int32_t *pos, cudaStream_t s);
cudaError_t launch_moe_gate_up(const uint8_t *w, int wt, int64_t expert_stride, int64_t n, int64_t k,
                               const uint16_t *xh, const uint16_t *xl, int64_t top_k, int64_t R, int64_t E,
                               const MoeWs &ws, uint8_t *hq, uint16_t *hbf, uint16_t *h16, uint16_t *h16lo,
                               int64_t hpitch, bool h16_grouped, cudaStream_t s);
cudaError_t launch_moe_down(const uint8_t *w, int wt, int64_t expert_stride, int64_t n, int64_t k,
                            const uint16_t *xh, const uint16_t *xl, int64_t top_k, int64_t R, int64_t E,
                            const MoeWs &ws, float *z, bool precise, cudaStream_t s, float *ysum = nullptr,
                            const float *route_w = nullptr);
// option "moe_deterministic" (default 1): 1 keeps the grouped down GEMM's
// per-route rows and sums each token's routes in slot order afterwards (the
// same bits on every run); 0 adds the weighted rows into the token rows with
// fp32 atomics in the GEMM's epilogue
int64_t option_moe_deterministic();
// y[R][n] (out dtype) from the per-route rows z, zero rows for skipped routes (pos < 0)
cudaError_t launch_moe_plain_store(const float *z, const int32_t *pos, const int32_t *ids, const int32_t *offsets,
                                   int64_t R, int64_t n, void *y, int yt, cudaStream_t s);
// y[T][n] = sum over each token's active routes of route_w * z row (in slot
// order); z rows in route order (offsets == nullptr) or in grouped order, route
// r at offsets[ids[r]] + pos[r]
cudaError_t launch_moe_finalize(const float *z, const int32_t *pos, const int32_t *ids, const int32_t *offsets,
                                const float *route_w, int64_t T, int64_t top_k, int64_t n, void *y, int yt,
                                cudaStream_t s);

}  // namespace gg
