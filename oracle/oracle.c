/*
 * CPU oracle for GGUF Q4_K / Q6_K / Q8_0 / IQ4_XS x Q8 integer matmul.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the bench's CPU
 * baseline leg may link, load or call this file. The CUDA library never does,
 * and this file shares no code, header, table or helper with it.
 *
 * Plain, slow, obviously correct: scalar loops, integer sub-block sums in
 * int64, every scale combine in double. Built with -O2 -ffp-contract=off so
 * that the one fp32 routine (the Q8 quantizer) runs exactly the IEEE
 * operations written here, one rounding each.
 *
 * What it computes (the sources):
 *  - xLLM v0.7 long-context article (Tencent Cloud), section 一 "背景":
 *    Q4_K / Q6_K weights are not dequantized to fp32; the kernel takes
 *    integer dot products against Q8-quantized activations and emits fp32.
 *  - same article, section B1.3: the Q8 activation quantization adds about
 *    0.5% RMS noise against the unquantized product and keeps the arg-max.
 *  - same article, section A2: a mixed model keeps attn_v and ffn_down in
 *    Q6_K, the other projections in Q4_K.
 *  - Agent Telemetry log, entry "批次化 MMVQ": the activation format is the
 *    q8_1 kind (int8 per 32 with a scale and a sum).
 *  - The pages name the Q4_K / Q6_K formats but never print their bit
 *    layout; the layout below is the public GGUF k-quant block layout,
 *    restated in words beside each decoder.
 *
 * Readings where the pages are silent (each applies in one place below):
 *  - Q8: d8 = amax/127 (IEEE fp32 divide), id = 1/d8 (0 if d8 == 0),
 *    q = clamp(roundf(x*id), -127, 127) with C roundf (ties away from zero),
 *    the clamp done in float (NaN -> 0, +-inf -> +-127) before the int
 *    conversion, s8 = d8 * (float)sum(q), one fp32 multiply. amax == 0 gives
 *    all zeros.
 *  - Q6_K "sub-block" for integer sums is the 16-weight scale group.
 *  - fp16 fields are IEEE binary16, little endian.
 */
#include "oracle.h"

#include <math.h>
#include <stdint.h>
#include <string.h>
#include <pthread.h>

/* Threads for the matmul routines. Output rows n are independent, so they
 * may be shared out among threads, row n to thread n mod T; every output is
 * still computed by one thread in the order written below, so the results
 * do not depend on the thread count. Returns the count in use. */
static int g_threads = 1;

int oracle_set_threads(int n)
{
    g_threads = n < 1 ? 1 : (n > 256 ? 256 : n);
    return g_threads;
}

struct mm_args {
    const uint8_t *W;
    const int8_t *codebook; /* IQ4_XS only */
    const int8_t *qs;
    const float *d8;
    int M, N, K;
    double *y, *absterm_out;
    int32_t *isum_out;
};

typedef void (*row_fn)(const struct mm_args *a, int n);

struct row_job {
    row_fn fn;
    const struct mm_args *a;
    int t, T;
};

static void *row_worker(void *p)
{
    const struct row_job *j = (const struct row_job *)p;
    for (int n = j->t; n < j->a->N; n += j->T) j->fn(j->a, n);
    return NULL;
}

/* fn(a, n) for every row n: on the calling thread, plus up to g_threads - 1
 * helper threads (a helper that cannot be started leaves its rows to the
 * calling thread). */
static void for_rows(row_fn fn, const struct mm_args *a)
{
    int T = g_threads < a->N ? g_threads : a->N;
    if (T <= 1) {
        for (int n = 0; n < a->N; n++) fn(a, n);
        return;
    }
    pthread_t th[256];
    int started[256];
    struct row_job jobs[256];
    for (int t = 0; t < T; t++) {
        jobs[t].fn = fn;
        jobs[t].a = a;
        jobs[t].t = t;
        jobs[t].T = T;
        started[t] = 0;
    }
    for (int t = 1; t < T; t++) started[t] = pthread_create(&th[t], NULL, row_worker, &jobs[t]) == 0;
    row_worker(&jobs[0]);
    for (int t = 1; t < T; t++) {
        if (started[t])
            pthread_join(th[t], NULL);
        else
            row_worker(&jobs[t]);
    }
}

static void zero_outputs(const struct mm_args *a)
{
    for (int m = 0; m < a->M; m++)
        for (int n = 0; n < a->N; n++) {
            a->y[(size_t)m * a->N + n] = 0.0;
            if (a->absterm_out) a->absterm_out[(size_t)m * a->N + n] = 0.0;
        }
}

/* IEEE 754 binary16 -> double, from the definition of the format:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent 0 is
 * subnormal (fraction * 2^-24), exponent 31 is inf/nan. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 31;
    int frac = h & 1023;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);
    }
    return sign ? -v : v;
}

static uint16_t read_u16le(const uint8_t *p)
{
    return (uint16_t)(p[0] | (p[1] << 8));
}

/* ---------------------------------------------------------------- Q8 */

/* Q8 activation quantization, one 32-block at a time, fp32 throughout.
 * x is [M][K] row-major; qs is [M][K]; d8 and s8 are [M][K/32]. */
int oracle_quantize_q8(const float *x, int M, int K,
                       int8_t *qs, float *d8, float *s8)
{
    if (M < 0 || K <= 0 || K % 32 != 0) return 1;
    int nblk = K / 32;
    for (int m = 0; m < M; m++) {
        for (int b = 0; b < nblk; b++) {
            const float *xb = x + (size_t)m * K + (size_t)b * 32;
            int8_t *qb = qs + (size_t)m * K + (size_t)b * 32;
            float amax = 0.0f;
            for (int i = 0; i < 32; i++) {
                float a = fabsf(xb[i]);
                if (a > amax) amax = a;
            }
            float d = amax / 127.0f;
            float id = (d != 0.0f) ? 1.0f / d : 0.0f;
            int isum = 0;
            for (int i = 0; i < 32; i++) {
                float t = xb[i] * id;
                float r = roundf(t);
                /* Saturate in float before converting: when amax is so small
                 * that 1/d8 overflows, x*id is +-inf (-> +-127) or 0*inf = NaN
                 * (-> 0); converting those to int directly is undefined. */
                if (r != r) r = 0.0f;
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                int q = (int)r;
                qb[i] = (int8_t)q;
                isum += q;
            }
            d8[(size_t)m * nblk + b] = d;
            s8[(size_t)m * nblk + b] = d * (float)isum;
        }
    }
    return 0;
}

/* ------------------------------------------------------------ SwiGLU */

/* The SwiGLU feed of the down projection, element by element in fp64 from
 * fp32 inputs: h = silu(g) * u, silu(g) = g * sigma(g) = g / (1 + e^-g)
 * (the gated activation between the gate/up and down matmuls of the layer
 * dispatch in the Agent Telemetry log). g -> -inf gives e^-g = inf and
 * h = +-0; g -> +inf gives h -> g * u. */
int oracle_silu_mul(const float *g, const float *u, int n, double *h)
{
    if (n < 0) return 1;
    for (int i = 0; i < n; i++) {
        double gi = (double)g[i];
        h[i] = gi / (1.0 + exp(-gi)) * (double)u[i];
    }
    return 0;
}

/* -------------------------------------------------------------- Q4_K */

/* Decode one Q4_K super-block (144 bytes, 256 weights) into its fields.
 * Layout (GGUF): d fp16 at byte 0, dmin fp16 at 2, 12 packed scale bytes at
 * 4..15, 128 quant bytes at 16..143.
 * The 12 scale bytes hold eight 6-bit scales sc[j] and eight 6-bit mins m[j]:
 *   j < 4 : sc = s[j] & 63,                         m = s[j+4] & 63
 *   j >= 4: sc = (s[j+4] & 15) | ((s[j-4] >> 6) << 4),
 *           m  = (s[j+4] >> 4) | ((s[j]   >> 6) << 4)
 * Quant byte 32*g + l (g = 0..3, l = 0..31) holds weight 64*g + l in its low
 * nibble and weight 64*g + 32 + l in its high nibble, so sub-block 2g is the
 * low nibbles of bytes 32g..32g+31 and sub-block 2g+1 their high nibbles. */
void oracle_q4k_fields(const uint8_t *blk, double *d, double *dmin,
                       int sc[8], int mn[8], int q[256])
{
    const uint8_t *s = blk + 4;
    const uint8_t *qb = blk + 16;
    *d = oracle_half_to_double(read_u16le(blk));
    *dmin = oracle_half_to_double(read_u16le(blk + 2));
    for (int j = 0; j < 8; j++) {
        if (j < 4) {
            sc[j] = s[j] & 63;
            mn[j] = s[j + 4] & 63;
        } else {
            sc[j] = (s[j + 4] & 15) | ((s[j - 4] >> 6) << 4);
            mn[j] = (s[j + 4] >> 4) | ((s[j] >> 6) << 4);
        }
    }
    for (int g = 0; g < 4; g++) {
        for (int l = 0; l < 32; l++) {
            uint8_t byte = qb[32 * g + l];
            q[64 * g + l] = byte & 15;
            q[64 * g + 32 + l] = byte >> 4;
        }
    }
}

/* Dequantize Q4_K rows to double: w = d*sc[j]*q - dmin*m[j] for the weight's
 * sub-block j. W is [N][K/256] super-blocks; w is [N][K]. */
int oracle_dequant_q4k(const uint8_t *W, int N, int K, double *w)
{
    if (N < 0 || K <= 0 || K % 256 != 0) return 1;
    int nsb = K / 256;
    for (int n = 0; n < N; n++) {
        for (int b = 0; b < nsb; b++) {
            const uint8_t *blk = W + ((size_t)n * nsb + b) * ORACLE_Q4K_BYTES;
            double d, dmin;
            int sc[8], mn[8], q[256];
            oracle_q4k_fields(blk, &d, &dmin, sc, mn, q);
            for (int i = 0; i < 256; i++) {
                int j = i / 32;
                w[(size_t)n * K + (size_t)b * 256 + i] =
                    d * sc[j] * q[i] - dmin * mn[j];
            }
        }
    }
    return 0;
}

/* -------------------------------------------------------------- Q6_K */

/* Decode one Q6_K super-block (210 bytes, 256 weights) into its fields.
 * Layout (GGUF): ql[128] at byte 0, qh[64] at 128, scales int8[16] at 192,
 * d fp16 at 208. For half h in {0,1} and l in 0..31, with L = ql + 64h and
 * H = qh + 32h, the 6-bit quants are
 *   weight 128h +      l = (L[l]    & 15) | (((H[l] >> 0) & 3) << 4)
 *   weight 128h + 32 + l = (L[l+32] & 15) | (((H[l] >> 2) & 3) << 4)
 *   weight 128h + 64 + l = (L[l]    >> 4) | (((H[l] >> 4) & 3) << 4)
 *   weight 128h + 96 + l = (L[l+32] >> 4) | (((H[l] >> 6) & 3) << 4)
 * Scale s[g] covers the 16 contiguous weights 16g..16g+15. */
void oracle_q6k_fields(const uint8_t *blk, double *d, int s[16], int q[256])
{
    const uint8_t *ql = blk;
    const uint8_t *qh = blk + 128;
    const int8_t *sc = (const int8_t *)(blk + 192);
    *d = oracle_half_to_double(read_u16le(blk + 208));
    for (int g = 0; g < 16; g++) s[g] = sc[g];
    for (int h = 0; h < 2; h++) {
        const uint8_t *L = ql + 64 * h;
        const uint8_t *H = qh + 32 * h;
        for (int l = 0; l < 32; l++) {
            q[128 * h + l]      = (L[l] & 15)      | (((H[l] >> 0) & 3) << 4);
            q[128 * h + 32 + l] = (L[l + 32] & 15) | (((H[l] >> 2) & 3) << 4);
            q[128 * h + 64 + l] = (L[l] >> 4)      | (((H[l] >> 4) & 3) << 4);
            q[128 * h + 96 + l] = (L[l + 32] >> 4) | (((H[l] >> 6) & 3) << 4);
        }
    }
}

/* Dequantize Q6_K rows to double: w = d*s[g]*(q - 32). */
int oracle_dequant_q6k(const uint8_t *W, int N, int K, double *w)
{
    if (N < 0 || K <= 0 || K % 256 != 0) return 1;
    int nsb = K / 256;
    for (int n = 0; n < N; n++) {
        for (int b = 0; b < nsb; b++) {
            const uint8_t *blk = W + ((size_t)n * nsb + b) * ORACLE_Q6K_BYTES;
            double d;
            int s[16], q[256];
            oracle_q6k_fields(blk, &d, s, q);
            for (int i = 0; i < 256; i++) {
                w[(size_t)n * K + (size_t)b * 256 + i] = d * s[i / 16] * (q[i] - 32);
            }
        }
    }
    return 0;
}

/* Q8_0 (xLLM v0.7 long-context article, section B3 + B4: symmetric int8,
 * one fp16 scale per 32 weights, no min term, 34-byte blocks). Public GGUF
 * block layout: d (fp16, little endian) at byte 0, then the 32 weights as
 * signed bytes at bytes 2..33; w = d * q. */
void oracle_q8_0_fields(const uint8_t *blk, double *d, int q[32])
{
    *d = oracle_half_to_double(read_u16le(blk));
    for (int i = 0; i < 32; i++) q[i] = (int8_t)blk[2 + i];
}

/* Dequantize Q8_0 rows to double. A row of K weights is K/32 blocks. */
int oracle_dequant_q8_0(const uint8_t *W, int N, int K, double *w)
{
    if (N < 0 || K <= 0 || K % 32 != 0) return 1;
    int nb = K / 32;
    for (int n = 0; n < N; n++) {
        for (int b = 0; b < nb; b++) {
            double d;
            int q[32];
            oracle_q8_0_fields(W + ((size_t)n * nb + b) * ORACLE_Q8_0_BYTES, &d, q);
            for (int i = 0; i < 32; i++) w[(size_t)n * K + (size_t)b * 32 + i] = d * q[i];
        }
    }
    return 0;
}

/* IQ4_XS (Agent Telemetry log, entries "找到" and "再一輪": 4-bit indices into
 * a 16-entry int8 codebook, kvalues_iq4nl, and a 32-weight sub-block laid out
 * like a Q4_0 block, low nibbles holding elements 0..15). The pages name the
 * codebook but do not print it, so it is an argument here (16 int8 values,
 * index order), not a table in this file. Public GGUF block layout, 136 bytes
 * per 256 weights:
 *   d (fp16, little endian) at byte 0; scales_h (uint16, little endian) at 2;
 *   scales_l[4] at 4; qs[128] at 8.
 * Sub-block j = 0..7 (32 weights) has the 6-bit scale
 *   ls_j = ((scales_l[j/2] >> 4*(j%2)) & 15) | (((scales_h >> 2j) & 3) << 4)
 * and weight i = 0..31 of it the index
 *   idx = (qs[16j + i%16] >> 4*(i/16)) & 15,
 * so w = d * (ls_j - 32) * codebook[idx]. */
void oracle_iq4xs_fields(const uint8_t *blk, const int8_t *codebook, double *d, int ls[8], int v[256])
{
    *d = oracle_half_to_double(read_u16le(blk));
    int sh = read_u16le(blk + 2);
    for (int j = 0; j < 8; j++) {
        int lo = (blk[4 + j / 2] >> (4 * (j % 2))) & 15;
        int hi = (sh >> (2 * j)) & 3;
        ls[j] = lo | (hi << 4);
        for (int i = 0; i < 32; i++) {
            int idx = (blk[8 + 16 * j + i % 16] >> (4 * (i / 16))) & 15;
            v[32 * j + i] = codebook[idx];
        }
    }
}

/* Dequantize IQ4_XS rows to double. */
int oracle_dequant_iq4xs(const uint8_t *W, const int8_t *codebook, int N, int K, double *w)
{
    if (N < 0 || K <= 0 || K % 256 != 0) return 1;
    int nsb = K / 256;
    double d;
    int ls[8], v[256];
    for (int n = 0; n < N; n++) {
        for (int b = 0; b < nsb; b++) {
            oracle_iq4xs_fields(W + ((size_t)n * nsb + b) * ORACLE_IQ4XS_BYTES, codebook, &d, ls, v);
            for (int i = 0; i < 256; i++)
                w[(size_t)n * K + (size_t)b * 256 + i] = d * (ls[i / 32] - 32) * v[i];
        }
    }
    return 0;
}

/* ----------------------------------------------------- integer route */

/* Q4_K x Q8 by integer sub-block sums (the route the kernels take).
 * For row n, token m, super-block b and sub-block j (32 weights):
 *   isum  = sum_i q[32j+i] * q8[m][256b+32j+i]            (exact, int64)
 *   isum8 = sum_i q8[m][256b+32j+i]                        (exact, int64)
 *   y[m][n] += d*sc_j*d8[m][8b+j]*isum - dmin*m_j*d8[m][8b+j]*isum8
 * All in double. isum_out (optional, [M][N][K/32]) receives isum.
 * absterm_out (optional, [M][N]) receives the sum of the absolute values of
 * every scaled term above, both the d-term and the dmin-term. */
static void q4k_row(const struct mm_args *A, int n)
{
    const int M = A->M, N = A->N, K = A->K;
    const int nsb = K / 256, nsub = K / 32;
    double d, dmin;
    int sc[8], mn[8], q[256];
    for (int b = 0; b < nsb; b++) {
        oracle_q4k_fields(A->W + ((size_t)n * nsb + b) * ORACLE_Q4K_BYTES, &d, &dmin, sc, mn, q);
        for (int m = 0; m < M; m++) {
            const int8_t *a = A->qs + (size_t)m * K + (size_t)b * 256;
            for (int j = 0; j < 8; j++) {
                int64_t isum = 0, isum8 = 0;
                for (int i = 0; i < 32; i++) {
                    isum += (int64_t)q[32 * j + i] * a[32 * j + i];
                    isum8 += a[32 * j + i];
                }
                double da = (double)A->d8[(size_t)m * nsub + 8 * b + j];
                double t1 = d * sc[j] * da * (double)isum;
                double t2 = dmin * mn[j] * da * (double)isum8;
                A->y[(size_t)m * N + n] += t1 - t2;
                if (A->absterm_out) A->absterm_out[(size_t)m * N + n] += fabs(t1) + fabs(t2);
                if (A->isum_out) A->isum_out[((size_t)m * N + n) * nsub + 8 * b + j] = (int32_t)isum;
            }
        }
    }
}

int oracle_matmul_q4k_q8(const uint8_t *W, const int8_t *qs, const float *d8,
                         int M, int N, int K,
                         double *y, double *absterm_out, int32_t *isum_out)
{
    if (M < 0 || N < 0 || K <= 0 || K % 256 != 0) return 1;
    struct mm_args A = {W, NULL, qs, d8, M, N, K, y, absterm_out, isum_out};
    zero_outputs(&A);
    for_rows(q4k_row, &A);
    return 0;
}

/* Q6_K x Q8 by integer sums over each 16-weight scale group g:
 *   isum_g = sum_i (q[16g+i] - 32) * q8[m][256b+16g+i]     (exact, int64)
 *   y[m][n] += d * s_g * d8[m][(256b+16g)/32] * isum_g     (double)
 * isum_out (optional) is [M][N][K/16]; absterm_out as for Q4_K. */
static void q6k_row(const struct mm_args *A, int n)
{
    const int M = A->M, N = A->N, K = A->K;
    const int nsb = K / 256, nsub = K / 32, ngrp = K / 16;
    double d;
    int s[16], q[256];
    for (int b = 0; b < nsb; b++) {
        oracle_q6k_fields(A->W + ((size_t)n * nsb + b) * ORACLE_Q6K_BYTES, &d, s, q);
        for (int m = 0; m < M; m++) {
            const int8_t *a = A->qs + (size_t)m * K + (size_t)b * 256;
            for (int g = 0; g < 16; g++) {
                int64_t isum = 0;
                for (int i = 0; i < 16; i++)
                    isum += (int64_t)(q[16 * g + i] - 32) * a[16 * g + i];
                double da = (double)A->d8[(size_t)m * nsub + 8 * b + g / 2];
                double t = d * s[g] * da * (double)isum;
                A->y[(size_t)m * N + n] += t;
                if (A->absterm_out) A->absterm_out[(size_t)m * N + n] += fabs(t);
                if (A->isum_out) A->isum_out[((size_t)m * N + n) * ngrp + 16 * b + g] = (int32_t)isum;
            }
        }
    }
}

int oracle_matmul_q6k_q8(const uint8_t *W, const int8_t *qs, const float *d8,
                         int M, int N, int K,
                         double *y, double *absterm_out, int32_t *isum_out)
{
    if (M < 0 || N < 0 || K <= 0 || K % 256 != 0) return 1;
    struct mm_args A = {W, NULL, qs, d8, M, N, K, y, absterm_out, isum_out};
    zero_outputs(&A);
    for_rows(q6k_row, &A);
    return 0;
}

/* Q8_0 x Q8 by integer block sums:
 *   isum = sum_i q[32j+i] * q8[m][32j+i]                   (exact, int64)
 *   y[m][n] += d_j * d8[m][j] * isum                        (double)
 * isum_out (optional) is [M][N][K/32]; absterm_out as for Q4_K. */
static void q8_0_row(const struct mm_args *A, int n)
{
    const int M = A->M, N = A->N, K = A->K;
    const int nb = K / 32;
    double d;
    int q[32];
    for (int j = 0; j < nb; j++) {
        oracle_q8_0_fields(A->W + ((size_t)n * nb + j) * ORACLE_Q8_0_BYTES, &d, q);
        for (int m = 0; m < M; m++) {
            const int8_t *a = A->qs + (size_t)m * K + (size_t)j * 32;
            int64_t isum = 0;
            for (int i = 0; i < 32; i++) isum += (int64_t)q[i] * a[i];
            double t = d * (double)A->d8[(size_t)m * nb + j] * (double)isum;
            A->y[(size_t)m * N + n] += t;
            if (A->absterm_out) A->absterm_out[(size_t)m * N + n] += fabs(t);
            if (A->isum_out) A->isum_out[((size_t)m * N + n) * nb + j] = (int32_t)isum;
        }
    }
}

int oracle_matmul_q8_0_q8(const uint8_t *W, const int8_t *qs, const float *d8,
                          int M, int N, int K,
                          double *y, double *absterm_out, int32_t *isum_out)
{
    if (M < 0 || N < 0 || K <= 0 || K % 32 != 0) return 1;
    struct mm_args A = {W, NULL, qs, d8, M, N, K, y, absterm_out, isum_out};
    zero_outputs(&A);
    for_rows(q8_0_row, &A);
    return 0;
}

/* IQ4_XS x Q8 by integer sub-block sums:
 *   isum_j = sum_i codebook[idx(32j+i)] * q8[m][256b+32j+i]   (exact, int64)
 *   y[m][n] += d * (ls_j - 32) * d8[m][8b+j] * isum_j          (double)
 * isum_out (optional) is [M][N][K/32]; absterm_out as for Q4_K. */
static void iq4xs_row(const struct mm_args *A, int n)
{
    const int M = A->M, N = A->N, K = A->K;
    const int nsb = K / 256, nsub = K / 32;
    double d;
    int ls[8], v[256];
    for (int b = 0; b < nsb; b++) {
        oracle_iq4xs_fields(A->W + ((size_t)n * nsb + b) * ORACLE_IQ4XS_BYTES, A->codebook, &d, ls, v);
        for (int m = 0; m < M; m++) {
            const int8_t *a = A->qs + (size_t)m * K + (size_t)b * 256;
            for (int j = 0; j < 8; j++) {
                int64_t isum = 0;
                for (int i = 0; i < 32; i++) isum += (int64_t)v[32 * j + i] * a[32 * j + i];
                double t = d * (ls[j] - 32) * (double)A->d8[(size_t)m * nsub + 8 * b + j] * (double)isum;
                A->y[(size_t)m * N + n] += t;
                if (A->absterm_out) A->absterm_out[(size_t)m * N + n] += fabs(t);
                if (A->isum_out) A->isum_out[((size_t)m * N + n) * nsub + 8 * b + j] = (int32_t)isum;
            }
        }
    }
}

int oracle_matmul_iq4xs_q8(const uint8_t *W, const int8_t *codebook, const int8_t *qs, const float *d8,
                           int M, int N, int K,
                           double *y, double *absterm_out, int32_t *isum_out)
{
    if (M < 0 || N < 0 || K <= 0 || K % 256 != 0) return 1;
    struct mm_args A = {W, codebook, qs, d8, M, N, K, y, absterm_out, isum_out};
    zero_outputs(&A);
    for_rows(iq4xs_row, &A);
    return 0;
}

/* ----------------------------------------------- straight dot products */

/* The plain definition: y[m][n] = sum_k w[n][k] * x[m][k], all double.
 * Used with x = d8*q8 (the dequantize-then-GEMV route the integer path
 * rearranges) and with x = the unquantized fp32 activation. */
int oracle_gemv_f64(const double *w, const double *x, int M, int N, int K, double *y)
{
    if (M < 0 || N < 0 || K < 0) return 1;
    for (int m = 0; m < M; m++) {
        for (int n = 0; n < N; n++) {
            double acc = 0.0;
            for (int k = 0; k < K; k++) acc += w[(size_t)n * K + k] * x[(size_t)m * K + k];
            y[(size_t)m * N + n] = acc;
        }
    }
    return 0;
}

/* Dequantized Q8 activation: xhat[m][k] = d8[m][k/32] * q8[m][k] (double). */
int oracle_dequant_q8(const int8_t *qs, const float *d8, int M, int K, double *xhat)
{
    if (M < 0 || K <= 0 || K % 32 != 0) return 1;
    for (int m = 0; m < M; m++)
        for (int k = 0; k < K; k++)
            xhat[(size_t)m * K + k] = (double)d8[(size_t)m * (K / 32) + k / 32] * qs[(size_t)m * K + k];
    return 0;
}
