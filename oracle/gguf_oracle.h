/*
 * gguf_oracle.h -- declarations of the scalar CPU oracle (test infrastructure
 * only; see gguf_oracle.c).  This header belongs to the oracle alone: the CUDA
 * library neither includes it nor shares any of its definitions.
 */
#ifndef GGUF_ORACLE_H
#define GGUF_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ggml type numbering (public GGUF convention) */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_Q4_0 = 2, ORC_Q4_1 = 3, ORC_Q5_0 = 6, ORC_Q5_1 = 7, ORC_Q8_0 = 8, ORC_Q8_1 = 9, ORC_Q4_K = 12, ORC_Q5_K = 13, ORC_Q6_K = 14, ORC_BF16 = 30,
       ORC_MXFP4 = 39 };

float orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_f16(float f);
float orc_bf16_to_f32(uint16_t h);
uint16_t orc_f32_to_bf16(float f);
uint16_t orc_f64_to_bf16(double f);

int64_t orc_block_elems(int type);
int64_t orc_block_bytes(int type);
int64_t orc_row_size(int type, int64_t k);
int64_t orc_sub_elems(int type);

void orc_quantize_q8_1_block(const float *x, uint8_t *out);
int orc_quantize_q8_1(const float *x, int64_t m, int64_t k, int64_t ldx, uint8_t *out);
int orc_quantize_weights(int type, const float *w, int64_t n, int64_t k, uint8_t *out);

int orc_dequantize_row(int type, const uint8_t *row, int64_t k, float *out);
int orc_dequantize_row_f64(int type, const uint8_t *row, int64_t k, double *out);
int orc_dequantize(int type, const uint8_t *w, int64_t rows, int64_t k, void *out, int ot);
int orc_get_rows(int type, const uint8_t *table, int64_t rows, int64_t k, const int32_t *ids, int64_t n_ids,
                 void *out, int ot);

int orc_block_dots(int type, const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, int32_t *sums);
int orc_mul_mat(int type, const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, double *y);
int orc_mul_mat_rows(int type, const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m, double *y,
                     int64_t n0, int64_t n1, int nthreads);
int orc_mul_mat_dequant_f64(int type, const uint8_t *w, int64_t n, int64_t k, const uint8_t *xq, int64_t m,
                            double *y);

int orc_moe_gate_up(int wt, const uint8_t *bank, int64_t n_experts, int64_t stride, int64_t two_i, int64_t h,
                    const uint8_t *xq, const int32_t *ids, int64_t n_tokens, int64_t top_k, float *hbuf, uint8_t *hq,
                    int64_t r0, int64_t r1, int nthreads);
int orc_moe_down(int wt, const uint8_t *bank, int64_t n_experts, int64_t stride, int64_t n_out, int64_t i_dim,
                 const uint8_t *hq, const int32_t *ids, const float *route_w, int64_t n_tokens, int64_t top_k,
                 double *y, int64_t t0, int64_t t1, int nthreads);

int orc_moe_plain(int wt, const uint8_t *bank, int64_t n_experts, int64_t stride, int64_t n, int64_t k,
                  const uint8_t *xq, const int32_t *ids, int64_t n_tokens, int64_t top_k, double *y);

#ifdef __cplusplus
}
#endif
#endif
