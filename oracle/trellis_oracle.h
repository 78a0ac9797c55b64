/* Declarations of the CPU oracle (test infrastructure only; see trellis_oracle.c). */
#ifndef TRELLIS_ORACLE_H
#define TRELLIS_ORACLE_H
#include <stdint.h>

float oracle_bf16_to_f32(uint16_t h);
uint16_t oracle_f32_to_bf16(float f);
uint32_t oracle_window(const uint32_t *blk, int t, int k, int L, int T);
int32_t oracle_code(uint32_t win);
float oracle_value(int32_t code);
uint16_t oracle_weight(const uint32_t *blk, int t, int k, int L, int T, uint16_t scale_bf16);
int oracle_check_geometry(int64_t K, int64_t N, int k, int L, int T);
int oracle_decode_rows(const uint32_t *codes, const uint16_t *scales, int64_t K, int64_t N,
                       int k, int L, int T, int64_t n0, int64_t n1, uint16_t *out);
int oracle_gemm_dense(const uint16_t *x, const uint16_t *W, int64_t M, int64_t K, int64_t nrows,
                      float *ref, double *refabs);
void oracle_silu_mul(const uint16_t *g, const uint16_t *u, int64_t n, uint16_t *act);

#endif
