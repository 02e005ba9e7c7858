/*
 * gguf_gb300.h -- C ABI of the GB300 (sm_103a) GGUF block-quantized matmul
 * library (libgguf_gb300.so).
 *
 * The library computes the hot path of a GGUF serving engine: activations in
 * fp32 / bf16 / fp16 are quantized to q8_1 blocks of 32 and multiplied against
 * Q8_0 / Q4_0 / Q4_K / Q5_K / Q6_K / MXFP4 weight blocks with per-block integer
 * dot products and an
 * fp32 scale / min combination; results come back in the activation dtype
 * with fp32 accumulation (FreeToken PR #690 "serve GGUF checkpoints on
 * vendored ggml-cuda kernels", section "Vendored ggml", list "What the ggml
 * patch changes").  The entry points are that page's op list: mul_mat,
 * mul_mat_id with the fused GLU and the MoE weighted sum, get_rows and
 * dequantize (same section, paragraph "Our own code next to it").
 *
 * Conventions shared by every entry point:
 *   - Pointers named w, x, xq, y, out, table, ids, ws are DEVICE pointers of
 *     the current CUDA device, owned by the caller.  The library allocates no
 *     device memory per call; scratch comes from the caller's workspace `ws`,
 *     sized by the matching *_ws_size query.
 *   - Every call is asynchronous and ordered on `stream` (a cudaStream_t;
 *     NULL is the legacy default stream).  No call synchronizes the host; in
 *     particular mul_mat_id groups its routes on the device and launches work
 *     only for the (expert, tile) pairs that have routes, without the host
 *     learning the counts (FreeToken PR #690, section "Vendored ggml").
 *   - Argument errors are reported synchronously as a status code; the
 *     library never aborts the process and never faults on bad arguments; the
 *     prior art turned such faults into errors (FreeToken issue #671 "MoE cache,
 *     CPU experts and GGUF support", section "Known issues").  gguf_last_error() returns a
 *     thread-local message for the last non-OK status.  CUDA launch errors
 *     come back as GGUF_ERR_CUDA.
 *   - Weight buffers must start on a 16-byte boundary.  Rows are packed back
 *     to back ([rows][row_size] bytes).  K must be a multiple of the type's
 *     block (32 for Q8_0 / Q4_0 / MXFP4 / q8_1, 256 for Q4_K / Q5_K / Q6_K: K-quant super-blocks span
 *     256 values, 1Cat-vLLM "GGUF on V100: implementation and acceptance control",
 *     section "TP/EP decision").  Offsets are 64-bit: no 2^31-block limit
 *     (FreeToken issue #671, "Known issues").  No kernel reads past the last
 *     byte of a weight view, so no tail padding is needed (unlike the MMQ tail
 *     read described in FreeToken PR #690, comment "GGUF experts in the offload
 *     slot cache have no MMQ tail padding").
 *
 * Block layouts (public GGUF convention; the pages name the formats but do not
 * print their bytes):
 *   Q8_0  34 B / 32 values : fp16 d, int8 q[32]                 v = d*q
 *   q8_1  36 B / 32 values : fp16 d, fp16 s = d*sum(q), int8 q[32]
 *   Q4_K 144 B / 256 values: fp16 d, fp16 dmin, 12 B of 6-bit (scale, min)
 *                            for 8 sub-blocks of 32, 128 B of 4-bit quants
 *                            v = d*scale_j*q - dmin*min_j
 *   Q6_K 210 B / 256 values: 128 B low 4 bits, 64 B high 2 bits, 16 int8
 *                            scales (sub-blocks of 16), fp16 d
 *                            v = d*scale_j*(q - 32)
 *   Q4_0  18 B / 32 values : fp16 d, 16 B of 4-bit quants (byte l: value l
 *                            low, value l + 16 high)            v = d*(q - 8)
 *   Q5_K 176 B / 256 values: Q4_K's 16-byte header, 32 B of fifth bits (value
 *                            i: bit i/32 of byte i%32), 128 B of low 4 bits
 *                            as Q4_K's quants            v = d*scale_j*q - dmin*min_j
 *   MXFP4 17 B / 32 values : E8M0 exponent e, 16 B of e2m1 codes in Q4_0's
 *                            order (OCP microscaling FP4)   v = e2m1(q)*2^(e-127)
 * Q4_0, Q5_K and MXFP4 are further tensor types the pages list (FreeToken PR
 * #690, "Tensor types"; transformers PR #45977, GgufLinear quant types).
 */
#ifndef GGUF_GB300_H
#define GGUF_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *gguf_stream_t; /* a cudaStream_t */

/* ggml type numbering (public GGUF convention). */
typedef enum {
    GGUF_F32 = 0,
    GGUF_F16 = 1,
    GGUF_Q4_0 = 2,
    GGUF_Q8_0 = 8,
    GGUF_Q8_1 = 9,
    GGUF_Q4_K = 12,
    GGUF_Q5_K = 13,
    GGUF_Q6_K = 14,
    GGUF_BF16 = 30,
    GGUF_MXFP4 = 39
} gguf_type;

typedef enum {
    GGUF_OK = 0,
    GGUF_ERR_INVALID_ARG = 1,      /* null pointer, negative size, bad mode/stride */
    GGUF_ERR_UNSUPPORTED_TYPE = 2, /* type not handled by this entry point */
    GGUF_ERR_SHAPE = 3,            /* K not a multiple of the block, or sizes inconsistent */
    GGUF_ERR_ALIGNMENT = 4,        /* a buffer or stride breaks the alignment rule */
    GGUF_ERR_WORKSPACE = 5,        /* ws smaller than the *_ws_size query */
    GGUF_ERR_CUDA = 6,             /* a CUDA runtime / launch error; see gguf_last_error() */
    GGUF_ERR_DEVICE = 7            /* a kernel gave up a bounded wait (gguf_device_errors) */
} gguf_status;

/* Thread-local message describing the last non-OK status of this thread. */
const char *gguf_last_error(void);

/* Values per block (1 for float types, 0 for unknown types). */
int64_t gguf_type_block_elems(int type);
/* Bytes per block (element size for float types, 0 for unknown types). */
int64_t gguf_type_block_bytes(int type);
/* Bytes of one row of k values ("ggml_row_size", FreeToken PR #690, comment on
 * MMQ tail padding); -1 if k is not a multiple of the block. */
int64_t gguf_row_size(int type, int64_t k);

/*
 * gguf_quantize_q8_1 -- activations to q8_1 (FreeToken PR #690, section
 * "Vendored ggml": fp32 / bf16 / fp16 activations go straight to q8_1).
 *   x   : [m][ldx] values of type xt (GGUF_F32, GGUF_BF16 or GGUF_F16); only
 *         the first k of each row are read.  ldx >= k.
 *   xq  : [m][k/32] q8_1 blocks (m * gguf_row_size(GGUF_Q8_1, k) bytes).
 * Per block of 32: d = amax/127 (IEEE fp32 division), q = roundf(x/d) (ties
 * away from zero; 0 when d == 0), s = fp16(d * sum(q)) with the fp32 d, and d
 * stored as fp16(d).  Bit-exact and deterministic.  |x| must stay below
 * 65504 * 127 so that d fits in fp16; NaN / Inf inputs give unspecified
 * blocks (no fault).  Requires k % 32 == 0.
 */
gguf_status gguf_quantize_q8_1(const void *x, int xt, int64_t m, int64_t k, int64_t ldx, void *xq,
                               gguf_stream_t stream);

/*
 * gguf_dequantize -- packed weights to float (FreeToken PR #690, op
 * "dequantize"; same-type float inputs are copied, types without a converter
 * are rejected: same page, summary of the later commits under "Validation").
 *   w   : [rows][row_size(wt, k)] bytes, wt in {Q8_0, Q4_0, Q4_K, Q5_K, Q6_K, MXFP4,
 *         Q8_1, F32, F16, BF16}
 *   out : [rows][k] of type ot in {F32, F16, BF16}
 * Values are computed in fp32 in the order  Q4_K, Q5_K: a = d*s; b = dmin*m;
 * a*q - b;  Q6_K: (d*sc)*(q-32);  Q8_0 / q8_1: d*q;  Q4_0: d*(q-8);  MXFP4:
 * 2^(e-128) * (2*e2m1(q)), negated for a code with the sign bit (so code 8
 * gives -0);  then rounded to ot with
 * round-to-nearest-even.  Bit-exact.  Float-to-float calls convert (RNE).
 */
gguf_status gguf_dequantize(const void *w, int wt, int64_t rows, int64_t k, void *out, int ot,
                            gguf_stream_t stream);

/*
 * gguf_get_rows -- out[i][:] = dequantize(table[ids[i]][:]) (FreeToken PR #690,
 * op "get_rows", used for the token embedding and the PLE table).
 *   table : [rows][row_size(tt, k)] bytes; ids : [n_ids] int32 device array;
 *   out   : [n_ids][k] of type ot (F32, F16, BF16).
 * An id outside [0, rows) yields a zero row (never an out-of-bounds read).
 */
gguf_status gguf_get_rows(const void *table, int tt, int64_t rows, int64_t k, const int32_t *ids, int64_t n_ids,
                          void *out, int ot, gguf_stream_t stream);

/*
 * gguf_mul_mat -- y[m][n] = sum_k W[n][k] * X[m][k] for a packed weight W
 * [n][k] (wt in {Q8_0, Q4_0, Q4_K, Q5_K, Q6_K, MXFP4}) and activations X [m][k].
 *   x  : [m][ldx] of type xt in {F32, BF16, F16} (quantized to q8_1 inside,
 *        into ws), or xt = GGUF_Q8_1: pre-quantized rows of row_size(Q8_1,k)
 *        bytes (ldx is then ignored) -- the way one q8_1 quantization serves
 *        several weight segments (FreeToken PR #690, section "Vendored ggml").
 *   y  : [m][ldy] of type yt in {F32, BF16, F16}; columns [0, n) of each row
 *        are written, so segments of a fused Linear can write column slices.
 *   ws : device workspace of at least gguf_mul_mat_ws_size(...) bytes
 *        (may be NULL when that size is 0).
 * Path: small m (<= option "mmvq_max_m", default 8; Q4_K up to option
 * "mmvq_tc_max_m", default 16) runs the bandwidth-bound MMVQ kernel
 * (exact int32 block sums from dp4a or int8 tensor-core MMAs, then the fp32
 * combination of the scales);
 * larger m runs the tensor-core MMQ kernel, which feeds tcgen05
 * fp16 operands (the exact fp32 block value of each weight and d16*q of each
 * activation) with fp32 accumulation: one fp16 operand per side for 16-bit
 * outputs (about 3e-4 of the row rms from the two roundings), hi + lo
 * operands on both sides for fp32 outputs (about 1e-6).
 */
size_t gguf_mul_mat_ws_size(int wt, int64_t n, int64_t k, int xt, int64_t m, int yt);
gguf_status gguf_mul_mat(const void *w, int wt, int64_t n, int64_t k, const void *x, int xt, int64_t m,
                         int64_t ldx, void *y, int yt, int64_t ldy, void *ws, size_t ws_bytes, gguf_stream_t stream);

/*
 * gguf_mul_mat_segments -- several weight matrices ("segments") that read the
 * same activations, e.g. the q/k/v or gate/up parts of a fused Linear:
 * y_s[m][n_s] = X . W_s^T for every segment s.  FreeToken PR #690 (section
 * "Vendored ggml") keeps one q8_1 quantization of the input for all segments;
 * here X is quantized once and, in the MMVQ range, one kernel launch covers
 * every segment (a row index runs through the segments in order).  The MMQ
 * range shares the quantized operand and runs one GEMM per segment.
 *   wt, k, x, xt, m, ldx, yt : as in gguf_mul_mat, common to all segments;
 *   segs[nseg]               : host array, 1 <= nseg <= GGUF_MAX_SEGMENTS; each
 *                              segment's w is 16-byte aligned [n][row_size(wt,k)]
 *                              bytes, y is [m][ldy] of type yt (columns [0, n)
 *                              written); n may be 0 (the segment is skipped).
 *   ws                       : gguf_mul_mat_segments_ws_size(...) bytes.
 * Errors as gguf_mul_mat; GGUF_ERR_INVALID_ARG for a bad segment count.
 */
#define GGUF_MAX_SEGMENTS 8
typedef struct gguf_segment {
    const void *w;  /* packed weight rows */
    int64_t n;      /* rows (output columns) */
    void *y;        /* output rows */
    int64_t ldy;    /* output row stride in elements (>= n) */
} gguf_segment;
size_t gguf_mul_mat_segments_ws_size(int wt, const gguf_segment *segs, int nseg, int64_t k, int xt, int64_t m,
                                     int yt);
gguf_status gguf_mul_mat_segments(int wt, const gguf_segment *segs, int nseg, int64_t k, const void *x, int xt,
                                  int64_t m, int64_t ldx, int yt, void *ws, size_t ws_bytes, gguf_stream_t stream);

/*
 * gguf_mul_mat_noalloc -- gguf_mul_mat for decode-sized products (m <= 8 rows
 * of float activations, k <= 16384), with no workspace argument and no device
 * allocation.  The pages have no counterpart of this entry point: it is for
 * callers that cannot hand over device memory at the call site, such as an
 * engine that launches from inside its own memory-pool callbacks, or one whose
 * allocator is not reachable from the code that issues the matmul.  The q8_1
 * copy of x lives in a fixed 256 KB device array inside this library instead
 * (m * k/32 * 36 bytes are used: 147,456 at the limits).
 *
 * Arguments, layouts and output are those of gguf_mul_mat with xt in
 * {F32, BF16, F16}; the result is the same MMVQ computation that gguf_mul_mat
 * runs for these sizes under the default options.
 * Errors: GGUF_ERR_WORKSPACE when m > 8 or k > 16384 (use gguf_mul_mat);
 * otherwise as gguf_mul_mat (m == 0 or n == 0 is a no-op; k == 0 with work
 * to do is GGUF_ERR_SHAPE).  Nothing has to be cleared between calls: every
 * scratch byte that is read was written by the same call.
 * The first call on each device looks up the scratch address; make it before
 * any stream capture.  The address is kept until the process exits and does
 * not survive cudaDeviceReset: do not call this entry point on a device after
 * resetting it.  The scratch is shared by every caller on the device:
 * calls that overlap in time (other streams, other host threads) race on it
 * and must be serialized by the caller.
 */
gguf_status gguf_mul_mat_noalloc(const void *w, int wt, int64_t n, int64_t k, const void *x, int xt, int64_t m,
                                 int64_t ldx, void *y, int yt, int64_t ldy, gguf_stream_t stream);

/*
 * gguf_copy_async -- dst[0, bytes) = src[0, bytes), stream-ordered.  Not a
 * step of the pages' method: the host <-> device staging that an engine
 * serving the decode step (FreeToken PR #690 "serve GGUF checkpoints on
 * vendored ggml-cuda kernels") puts around it.  The copy runs on the SMs as a
 * programmatic dependent launch, so it stays in the chain of the path's
 * launches instead of ending it the way a copy-engine copy does.
 *   dst, src : device, managed or pinned (page-locked) host memory, any
 *              alignment (16-byte aligned pointers move 16 bytes per load);
 *              the ranges may not overlap.  The caller keeps both alive until
 *              the stream has passed the copy.
 *   bytes    : >= 0 (0 is a no-op).
 * Errors: GGUF_ERR_INVALID_ARG for a negative size, a null pointer,
 * overlapping ranges or a buffer that is not device-accessible (pageable host
 * memory is refused before anything is launched); GGUF_ERR_CUDA for a launch
 * error.
 */
gguf_status gguf_copy_async(void *dst, const void *src, int64_t bytes, gguf_stream_t stream);

/*
 * gguf_mul_mat_batch -- several decode-sized products of one weight type and
 * K in one call, each a gguf_mul_mat_segments on q8_1 rows that were written
 * before the call: job j computes y_s[m_j][n_s] = Xq_j . W_s^T for its
 * segments.  The pages' decode step issues one MMVQ per weight (FreeToken PR
 * #690, section "Vendored ggml", MMVQ for small batches); a batch of such
 * products is launched as one chain of kernels (programmatic dependent launch)
 * in which each kernel after the first starts as the previous one drains, so
 * the GPU pays the start-up and tail of a launch once for the batch.
 *   jobs[njobs] : host array, njobs <= GGUF_MAX_BATCH_JOBS; each job's xq is
 *                 [m][row_size(GGUF_Q8_1, k)] bytes (4-byte aligned) and its
 *                 m is decode-sized (the MMVQ range of gguf_mul_mat: at most
 *                 option "mmvq_max_m" rows, Q4_K up to "mmvq_tc_max_m");
 *                 segments as in gguf_mul_mat_segments.
 * The jobs run concurrently: no job may write memory that another job of the
 * batch reads or writes (its y may not be another job's xq).  The call ends
 * with an ordinary launch, so work queued after it sees every job complete.
 * No workspace.  Errors as gguf_mul_mat_segments; GGUF_ERR_INVALID_ARG for a
 * job outside the MMVQ range; nothing is launched unless every job is valid.
 */
#define GGUF_MAX_BATCH_JOBS 8
typedef struct gguf_mm_job {
    const gguf_segment *segs;  /* host array of the job's weight segments */
    int nseg;                  /* 1 .. GGUF_MAX_SEGMENTS */
    const void *xq;            /* q8_1 activation rows */
    int64_t m;                 /* rows of xq */
} gguf_mm_job;
gguf_status gguf_mul_mat_batch(int wt, int64_t k, const gguf_mm_job *jobs, int njobs, int yt, gguf_stream_t stream);

/*
 * gguf_mul_mat_batch_typed -- gguf_mul_mat_batch with the weight type and K
 * given per job, so products of different types on one input (a layer's q
 * and k in Q4_K and its v in Q6_K, all on the attention input) run in one
 * chain and none waits for another.  Same rules and errors as
 * gguf_mul_mat_batch, checked per job (GGUF_ERR_UNSUPPORTED_TYPE /
 * GGUF_ERR_SHAPE name the job); one output type yt for all jobs.
 */
typedef struct gguf_mm_job_typed {
    int wt;                    /* the job's weight type */
    int64_t k;                 /* the job's K */
    const gguf_segment *segs;  /* host array of the job's weight segments */
    int nseg;                  /* 1 .. GGUF_MAX_SEGMENTS */
    const void *xq;            /* q8_1 activation rows, [m][row_size(GGUF_Q8_1, k)] */
    int64_t m;                 /* rows of xq */
} gguf_mm_job_typed;
gguf_status gguf_mul_mat_batch_typed(const gguf_mm_job_typed *jobs, int njobs, int yt, gguf_stream_t stream);

/* mul_mat_id modes */
#define GGUF_MOE_GATE_UP_SWIGLU 0   /* h[r] = silu(gate) * up, rounded to bf16, out as BF16 or Q8_1 */
#define GGUF_MOE_DOWN_WEIGHTED_SUM 1 /* y[t] = sum_k route_w[t][k] * (W[e] . x[route]) */
#define GGUF_MOE_PLAIN 2             /* y[route] = W[e] . x[token]: one row per route, no weighting */

/*
 * Arguments of gguf_mul_mat_id (MoE experts).
 *   w, wt           : expert bank base; expert e's packed [n][k] matrix starts at
 *                     w + e * expert_stride bytes (a flat [n_experts, stride]
 *                     bank as in FreeToken PR #196's bank geometry discussion);
 *                     expert_stride >= n * row_size and a multiple of 16.
 *   n, k            : rows and columns of one expert matrix.  GATE_UP: n = 2*I,
 *                     gate rows [0, I) first, then up rows [I, 2I) (the merged
 *                     gate_up layout of transformers PR #45977 "GgufExperts").
 *   x, xt, ldx      : GATE_UP: token rows [n_tokens][ldx] (F32 / BF16 / F16) or
 *                     q8_1 rows [n_tokens][row_size(Q8_1, k)];
 *                     DOWN: route rows [n_tokens * top_k][ldx] (BF16) or q8_1
 *                     rows [n_tokens * top_k][row_size(Q8_1, k)], route
 *                     r = t * top_k + j.
 *                     PLAIN: token rows as for GATE_UP; every route of token
 *                     t reads row t.
 *   ids             : [n_tokens][top_k] int32 expert ids; id < 0 or >= n_experts
 *                     marks an inactive route (skipped, never read), and a token
 *                     may name the same expert more than once (FreeToken issue
 *                     #671, "Known issues").
 *   route_w         : [n_tokens][top_k] fp32 weights (DOWN; NULL means 1.0).
 *                     A route whose weight is 0 is skipped.  PLAIN ignores it.
 *   y, yt           : GATE_UP: [n_tokens * top_k][n/2] of yt = BF16, Q8_1 (q8_1
 *                     rows of row_size(Q8_1, n/2) bytes) or F16 (the dequantized
 *                     q8_1 values d16*q, the form the down GEMM consumes);
 *                     inactive routes get zero rows.  n must be a multiple of 128.
 *                     DOWN: [n_tokens][n] of yt = F32, BF16 or F16.
 *                     PLAIN: [n_tokens * top_k][n] of yt = F32, BF16 or F16,
 *                     row r = t * top_k + j; inactive routes get zero rows.
 *                     (The generic mul_mat_id without a fused epilogue, for
 *                     experts whose output the caller combines itself.)
 *   workspace       : 256-byte aligned, gguf_mul_mat_id_ws_size(args) bytes.
 *   dev_status      : optional device int32; the count of ids >= n_experts is
 *                     added to it (never a trap, never a host sync).
 * The intermediate h is kept in the activation dtype (bf16) and then quantized
 * to q8_1 (FreeToken PR #690, section "Changes": the intermediates stay in the
 * activation dtype).
 * Path: up to option "moe_vec_max_tokens" tokens (default 256) the call runs
 * the route-batched MMVQ (one launch over all route slots, each reading its
 * expert's rows once with exact int32 block sums; FreeToken PR #690, section
 * "Changes": MoE takes MMVQ for small batches and MMQ above, with the
 * grouped-MMQ-vs-vec crossover at 16 tokens on sm_120 in FreeToken PR #196,
 * "Dispatch thresholds"), else the tensor-core grouped GEMM over the (expert,
 * 128-route tile) pairs that hold routes.  Rows longer than 16384
 * values (8192 for Q8_0) always take the grouped GEMM.
 */
typedef struct {
    const void *w;
    int wt;
    int64_t n_experts;
    int64_t expert_stride;
    int64_t n;
    int64_t k;
    const void *x;
    int xt;
    int64_t n_tokens;
    int64_t ldx;
    const int32_t *ids;
    int64_t top_k;
    const float *route_w;
    int mode;
    void *y;
    int yt;
    int32_t *dev_status;
} gguf_moe_args;

size_t gguf_mul_mat_id_ws_size(const gguf_moe_args *args);
gguf_status gguf_mul_mat_id(const gguf_moe_args *args, void *ws, size_t ws_bytes, gguf_stream_t stream);

/*
 * gguf_moe_ffn -- the whole MoE expert block in one call: q8_1 quantization of
 * the token rows, gate_up mul_mat_id with the fused SwiGLU (h kept in bf16,
 * then quantized to q8_1), and the down mul_mat_id with the fused
 * expert-weighted sum.  One device-side route grouping serves both GEMMs and
 * the intermediate stays in the workspace.  Same conventions as
 * gguf_mul_mat_id; banks hold [2*inter][hidden] (gate rows, then up rows) and
 * [hidden][inter] matrices per expert.  y : [n_tokens][hidden] of yt (F32, BF16
 * or F16).  Routes with weight 0 are skipped by both GEMMs.  The same
 * "moe_vec_max_tokens" option selects the route-batched MMVQ for both products.
 */
typedef struct {
    const void *w_gate_up;
    int gate_up_type;
    int64_t gate_up_stride;
    const void *w_down;
    int down_type;
    int64_t down_stride;
    int64_t n_experts;
    int64_t hidden;
    int64_t inter;
    const void *x;
    int xt;
    int64_t n_tokens;
    int64_t ldx;
    const int32_t *ids;
    int64_t top_k;
    const float *route_w;
    void *y;
    int yt;
    int32_t *dev_status;
} gguf_moe_ffn_args;

size_t gguf_moe_ffn_ws_size(const gguf_moe_ffn_args *args);
gguf_status gguf_moe_ffn(const gguf_moe_ffn_args *args, void *ws, size_t ws_bytes, gguf_stream_t stream);

/*
 * gguf_debug_block_dots -- test hook: the exact int32 dot product of every
 * weight sub-block (32 values for Q8_0 / Q4_0 / Q4_K / Q5_K / MXFP4, 16 for Q6_K;
 * Q4_0 and Q6_K quants enter with their offsets 8 and 32 subtracted, MXFP4
 * codes as 2 * e2m1) with the matching
 * q8_1 activation quants.  sums : [m][n][k / sub] int32.  Bit-exact.
 */
gguf_status gguf_debug_block_dots(const void *w, int wt, int64_t n, int64_t k, const void *xq, int64_t m,
                                  int32_t *sums, gguf_stream_t stream);

/*
 * Tunables (host-global, not thread-safe against concurrent calls):
 *   "mmvq_max_m"  : largest m routed to MMVQ (default 8; FreeToken issue #671,
 *                   "Known issues": MMQ takes over above 8 tokens).
 *   "mmq_enable"  : 0 routes every m through MMVQ (default 1).
 *   "mmvq_tc"     : 1 (default) lets mmvq_tc_min_m..8 tokens of Q4_K rows
 *                   (n >= 2048) run the tensor-core MMVQ; 0 keeps them on the
 *                   dp4a MMVQ.
 *   "mmvq_tc_min_m": fewest tokens that take the tensor-core MMVQ, 1 .. 8
 *                   (default 5).
 *   "moe_vec_max_tokens": mul_mat_id / moe_ffn calls of at most this many
 *                   tokens take the route-batched MMVQ; 0 .. 256, default 256
 *                   (measured on GB300 for the E=256, top-8 expert block:
 *                   4-6x faster than the grouped GEMM at 1..16 tokens,
 *                   2.3x at 128, still 1.3x at 256).
 *   "mmvq_tc_max_m": Q4_K products of 9 up to this many tokens stay on the
 *                   tensor-core MMVQ (2 or 4 n-tiles of 8 tokens) instead
 *                   of MMQ; 8 .. 32, default 16 (the measured crossover on
 *                   GB300: 4 n-tiles are not faster than MMQ).
 *   "mmq_stage"   : 1 (default) lets the tensor-core GEMMs (MMQ and the
 *                   grouped MoE GEMMs) stage packed weight rows in shared
 *                   memory by bulk tensor copies where the rows' layout allows
 *                   it; 0 has the producer warps load them from global memory.
 *   "mmq_bn_max"  : widest activation tile of the dense MMQ, 128 or 256
 *                   (default 256).  Tiles of at most 128 rows keep the weight
 *                   operand in tensor memory.
 *   "mmq_split_k" : 1 (default) lets MMQ calls with few output tiles split K
 *                   across CTAs (fp32 partial sums, then one conversion).
 *   "moe_deterministic": 1 (default) keeps the grouped down GEMM's per-route
 *                   rows and sums each token's routes in slot order afterwards
 *                   (the same bits on every run); 0 adds the weighted rows into
 *                   fp32 token rows inside the GEMM's epilogue (bulk
 *                   reduce-adds, or fp32 atomics when n % 4 != 0), whose
 *                   summation order varies from run to run.
 *   "moe_down_precise": 1 runs the grouped down GEMM on hi + lo operands for
 *                   16-bit outputs too (fp32 outputs always do); default 0.
 *   "moe_gate_up_precise": 1 (default) runs the grouped gate_up GEMM on hi + lo
 *                   operands (three MMAs per K step); 0 on one fp16 operand
 *                   per side.
 *   "mmq_engine"  : 0 (default) runs the prefill (MMQ-range) products on the
 *                   fused tensor-core MMQ; 1 runs those with BF16 / F16
 *                   outputs as dequantize (weights -> fp16) + one library GEMM
 *                   (cuBLAS, opened at run time: GGUF_ERR_CUDA when it cannot
 *                   be loaded) on the activations' fp16 q8_1 operand, the
 *                   alternative engine FreeToken PR #196 ("Gains") races
 *                   against MMQ.  Its workspace adds n * k * 2 bytes (the
 *                   fp16 weights) and, for BF16 outputs, m * n * 4 (the GEMM
 *                   writes fp32 rows that one pass converts), and its min
 *                   terms use d_a * sum(q) instead
 *                   of the stored s_a (about 1e-3 of the row rms), within
 *                   the 16-bit output bound.  FP32 outputs keep the fused
 *                   MMQ.
 * Returns GGUF_ERR_INVALID_ARG for an unknown key or a value out of range.
 */
gguf_status gguf_set_option(const char *key, int64_t value);
int64_t gguf_get_option(const char *key);

/*
 * gguf_device_errors -- the error word of the tensor-core kernels (MMQ and the
 * grouped MoE GEMMs) on the current device.  Those kernels bound every wait
 * of their pipeline (one second); a CTA whose wait gives up sets the bit of
 * its role, stops its work and exits, so the call that launched it has
 * already returned GGUF_OK while its output is incomplete.  The prior art
 * turned faults into errors the caller can see (FreeToken issue #671 "MoE
 * cache, CPU experts and GGUF support", section "Known issues"); this query is
 * how such a timeout reaches the caller.
 *   flags  : host int32; receives the word (0 when every kernel finished).
 *   clear  : nonzero resets the word to 0 after reading it.
 *   stream : the word is read after all work queued on `stream` (the call
 *            synchronizes that stream).
 * Returns GGUF_OK when the word is 0, GGUF_ERR_DEVICE when a bit is set (the
 * message names the roles: 1 operand loads, 2 MMA issue, 4 weight unpack,
 * 8 epilogue, 16 accumulator hand-over, 32 packed-weight loads),
 * GGUF_ERR_INVALID_ARG for a null flags pointer.
 *
 * gguf_device_errors_async -- the same read (and optional reset) as a
 * stream-ordered device step with no host synchronization: the word is
 * written to the device int32 *dev_flags when the stream reaches it.  Usable
 * inside CUDA graph capture.
 */
gguf_status gguf_device_errors(int32_t *flags, int clear, gguf_stream_t stream);
gguf_status gguf_device_errors_async(int32_t *dev_flags, int clear, gguf_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* GGUF_GB300_H */
