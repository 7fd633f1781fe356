/*
 * CPU oracle for GGUF Q4_K / Q6_K / Q8_0 / IQ4_XS x Q8 integer matmul.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
 * baseline leg may use it. It shares nothing with the CUDA library.
 *
 * Layouts (all row-major, host memory, caller-owned):
 *   x   fp32 [M][K]            unquantized activations
 *   qs  int8 [M][K]            Q8 quants
 *   d8  fp32 [M][K/32]         Q8 block scales
 *   s8  fp32 [M][K/32]         Q8 block scale * block sum of quants
 *   W   bytes [N][K/256][144]  Q4_K super-blocks, [N][K/256][210] Q6_K,
 *                              [N][K/256][136] IQ4_XS, or [N][K/32][34] Q8_0
 *   codebook int8 [16]         IQ4_XS value of each 4-bit index
 *   y   double [M][N]
 * Every function returns 0 on success, 1 on a bad shape.
 */
#ifndef XQ_ORACLE_H
#define XQ_ORACLE_H

#include <stdint.h>

#define ORACLE_Q4K_BYTES 144
#define ORACLE_Q6K_BYTES 210
#define ORACLE_Q8_0_BYTES 34
#define ORACLE_IQ4XS_BYTES 136

#ifdef __cplusplus
extern "C" {
#endif

double oracle_half_to_double(uint16_t h);

int oracle_quantize_q8(const float *x, int M, int K,
                       int8_t *qs, float *d8, float *s8);

/* h[i] = silu(g[i]) * u[i] in fp64, silu(g) = g / (1 + e^-g). */
int oracle_silu_mul(const float *g, const float *u, int n, double *h);

void oracle_q4k_fields(const uint8_t *blk, double *d, double *dmin,
                       int sc[8], int mn[8], int q[256]);
void oracle_q6k_fields(const uint8_t *blk, double *d, int s[16], int q[256]);
void oracle_q8_0_fields(const uint8_t *blk, double *d, int q[32]);
void oracle_iq4xs_fields(const uint8_t *blk, const int8_t *codebook, double *d, int ls[8], int v[256]);

int oracle_dequant_q4k(const uint8_t *W, int N, int K, double *w);
int oracle_dequant_q6k(const uint8_t *W, int N, int K, double *w);
int oracle_dequant_q8_0(const uint8_t *W, int N, int K, double *w);
int oracle_dequant_iq4xs(const uint8_t *W, const int8_t *codebook, int N, int K, double *w);
int oracle_dequant_q8(const int8_t *qs, const float *d8, int M, int K, double *xhat);

int oracle_matmul_q4k_q8(const uint8_t *W, const int8_t *qs, const float *d8,
                         int M, int N, int K,
                         double *y, double *absterm_out, int32_t *isum_out);
int oracle_matmul_q6k_q8(const uint8_t *W, const int8_t *qs, const float *d8,
                         int M, int N, int K,
                         double *y, double *absterm_out, int32_t *isum_out);

int oracle_matmul_q8_0_q8(const uint8_t *W, const int8_t *qs, const float *d8,
                          int M, int N, int K,
                          double *y, double *absterm_out, int32_t *isum_out);

int oracle_matmul_iq4xs_q8(const uint8_t *W, const int8_t *codebook, const int8_t *qs, const float *d8,
                           int M, int N, int K,
                           double *y, double *absterm_out, int32_t *isum_out);

int oracle_gemv_f64(const double *w, const double *x, int M, int N, int K, double *y);

/* Threads for the matmul routines (OpenMP over output rows when built with
 * it; results do not depend on the count). Returns the count in use. */
int oracle_set_threads(int n);

#ifdef __cplusplus
}
#endif

#endif
