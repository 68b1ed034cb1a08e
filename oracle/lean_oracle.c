/*
 * lean_oracle.c -- plain, slow, scalar fp64 CPU oracle for the block-quantized
 * weight x activation product.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library.  The product (the
 * CUDA library) shares no code, header, table or helper with it, and nothing in
 * the product calls it.
 *
 * What it computes (the plain definition, no blocking or reordering):
 *
 *     w[n,k]   = the exact value of weight (n,k) decoded from its block
 *     y[m,n]   = sum_k w[n,k] * x[m,k]          (fp64)
 *     B[m,n]   = sum_k |w[n,k] * x[m,k]|         (fp64, the tolerance scale)
 *
 * Sources for the formats:
 *   - "lean" README (llm-web), model table: Q4_0 weights, Q6_K embedding, and
 *     the Q8_0 GGUF checkpoints of its parity tests.
 *   - "oxinfer" crate page, "How it works", quant.rs bullet: Q4_0 is two nibbles
 *     per byte with an f16 scale per 32 weights; Q8 is 32 weights per scale.
 *   - "oxinfer" crate page, "Pre-quantized checkpoints": quantized matrices are
 *     kept as a quant plane plus a scale plane.
 *   - "wgpu-llm" README, "INT8 mode": symmetric INT8 with block size 64.
 *   The pages fix neither the byte order of the nibbles nor the Q6_K bit layout;
 *   this file takes the GGUF block layouts as the reading (stated per format
 *   below).  The value laws are d*(q-8) (Q4_0), d*q (Q8_0, INT8-B64) and
 *   d*sc*(q-32) (Q6_K).
 *
 * Canonical (interchange) block layouts, little-endian:
 *   Q4_0     18 B / 32 weights : [d fp16][qs 16 B]; element j<16 is the low
 *                                nibble of qs[j], element j+16 its high nibble.
 *   Q8_0     34 B / 32 weights : [d fp16][32 x int8]
 *   INT8-B64 66 B / 64 weights : [d fp16][64 x int8]
 *   Q6_K    210 B / 256 weights: [ql 128 B][qh 64 B][sc 16 x int8][d fp16]
 * Blocks run along K inside a row; row n of W is K/block_elems consecutive
 * blocks.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_Q4_0 = 0, ORACLE_Q8_0 = 1, ORACLE_I8_B64 = 2, ORACLE_Q6_K = 3 };

/* IEEE 754 binary16 -> double, written out from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.  Exponent 0 is the
 * subnormal range (no hidden bit, scale 2^-14); exponent 31 is Inf / NaN. */
double oracle_fp16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);               /* f * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

int oracle_block_elems(int fmt)
{
    switch (fmt) {
    case ORACLE_Q4_0: return 32;
    case ORACLE_Q8_0: return 32;
    case ORACLE_I8_B64: return 64;
    case ORACLE_Q6_K: return 256;
    }
    return 0;
}

int oracle_block_bytes(int fmt)
{
    switch (fmt) {
    case ORACLE_Q4_0: return 2 + 16;
    case ORACLE_Q8_0: return 2 + 32;
    case ORACLE_I8_B64: return 2 + 64;
    case ORACLE_Q6_K: return 128 + 64 + 16 + 2;
    }
    return 0;
}

static uint16_t read_u16le(const uint8_t *p) { return (uint16_t)(p[0] | (p[1] << 8)); }

/* Value of element j of one canonical block. */
static double block_value(int fmt, const uint8_t *blk, int j)
{
    switch (fmt) {
    case ORACLE_Q4_0: {
        double d = oracle_fp16_to_double(read_u16le(blk));
        const uint8_t *qs = blk + 2;
        int q = (j < 16) ? (qs[j] & 0x0f) : (qs[j - 16] >> 4);
        return d * (double)(q - 8);
    }
    case ORACLE_Q8_0:
    case ORACLE_I8_B64: {
        double d = oracle_fp16_to_double(read_u16le(blk));
        int q = (int)(int8_t)blk[2 + j];
        return d * (double)q;
    }
    case ORACLE_Q6_K: {
        const uint8_t *ql = blk;
        const uint8_t *qh = blk + 128;
        const int8_t *sc = (const int8_t *)(blk + 192);
        double d = oracle_fp16_to_double(read_u16le(blk + 208));
        int h = j / 128;          /* which half of the super-block      */
        int e = j % 128;          /* position inside that half          */
        int g = e / 32;           /* 32-element group inside the half   */
        int l = e % 32;
        /* low 4 bits: nibble g/2 of ql[64h + 32*(g%2) + l]             */
        int lo = (ql[64 * h + 32 * (g % 2) + l] >> (4 * (g / 2))) & 0x0f;
        /* high 2 bits: bits 2g, 2g+1 of qh[32h + l]                     */
        int hi = (qh[32 * h + l] >> (2 * g)) & 0x03;
        int q = lo | (hi << 4);
        /* one int8 sub-scale per 16 consecutive elements                */
        return d * (double)sc[j / 16] * (double)(q - 32);
    }
    }
    return NAN;
}

/* Decode one row of canonical blocks (K weights) into w[0..K). */
int oracle_dequant_row(int fmt, const uint8_t *row, int64_t K, double *w)
{
    int be = oracle_block_elems(fmt), bb = oracle_block_bytes(fmt);
    if (be == 0 || K % be != 0) return -1;
    for (int64_t k = 0; k < K; ++k)
        w[k] = block_value(fmt, row + (k / be) * bb, (int)(k % be));
    return 0;
}

/* w[N][K] fp64 for the whole matrix. */
int oracle_dequant(int fmt, const uint8_t *W, int64_t N, int64_t K, double *w)
{
    int be = oracle_block_elems(fmt), bb = oracle_block_bytes(fmt);
    if (be == 0 || K % be != 0) return -1;
    int64_t row_bytes = (K / be) * bb;
    for (int64_t n = 0; n < N; ++n)
        if (oracle_dequant_row(fmt, W + n * row_bytes, K, w + n * K)) return -1;
    return 0;
}

/* ---- y = W x over all (m, n), rows split across threads for timing ---- */

typedef struct {
    int fmt;
    const uint8_t *W;
    const float *x;
    double *y, *bound;
    int64_t N, K, M, n0, n1;
    int status;
} job_t;

static void *row_range(void *arg)
{
    job_t *j = (job_t *)arg;
    int be = oracle_block_elems(j->fmt), bb = oracle_block_bytes(j->fmt);
    int64_t row_bytes = (j->K / be) * bb;
    double *w = (double *)malloc(sizeof(double) * (size_t)j->K);
    if (!w) { j->status = -2; return NULL; }
    for (int64_t n = j->n0; n < j->n1; ++n) {
        oracle_dequant_row(j->fmt, j->W + n * row_bytes, j->K, w);
        for (int64_t m = 0; m < j->M; ++m) {
            const float *xm = j->x + m * j->K;
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < j->K; ++k) {
                double p = w[k] * (double)xm[k];
                acc += p;
                mag += fabs(p);
            }
            j->y[m * j->N + n] = acc;
            if (j->bound) j->bound[m * j->N + n] = mag;
        }
    }
    free(w);
    j->status = 0;
    return NULL;
}

/* y[M][N] (and bound[M][N] if non-null) from canonical W[N][K/be blocks] and
 * x[M][K] fp32.  n_threads <= 1 runs on the calling thread. Returns 0 on
 * success, -1 on a bad shape or format, -2 on allocation failure. */
int oracle_qmatmul(int fmt, const uint8_t *W, const float *x, double *y, double *bound,
                   int64_t N, int64_t K, int64_t M, int n_threads)
{
    int be = oracle_block_elems(fmt);
    if (be == 0 || N < 0 || M < 0 || K <= 0 || K % be != 0) return -1;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > N) n_threads = N > 0 ? (int)N : 1;
    job_t *jobs = (job_t *)calloc((size_t)n_threads, sizeof(job_t));
    pthread_t *tids = (pthread_t *)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return -2; }
    for (int t = 0; t < n_threads; ++t) {
        job_t j = {fmt, W, x, y, bound, N, K, M, N * t / n_threads, N * (t + 1) / n_threads, -3};
        jobs[t] = j;
    }
    int status = 0;
    if (n_threads == 1) {
        row_range(&jobs[0]);
        status = jobs[0].status;
    } else {
        for (int t = 0; t < n_threads; ++t)
            if (pthread_create(&tids[t], NULL, row_range, &jobs[t])) { jobs[t].status = -2; tids[t] = 0; }
        for (int t = 0; t < n_threads; ++t) {
            if (tids[t]) pthread_join(tids[t], NULL);
            if (jobs[t].status) status = jobs[t].status;
        }
    }
    free(jobs);
    free(tids);
    return status;
}

/* Selected outputs only: for each i < P, y[i] and bound[i] for the pair
 * (m_idx[i], n_idx[i]).  Used to check sampled outputs of full-size runs. */
int oracle_qmatmul_pairs(int fmt, const uint8_t *W, const float *x, int64_t N, int64_t K, int64_t M,
                         int64_t P, const int64_t *m_idx, const int64_t *n_idx, double *y, double *bound)
{
    int be = oracle_block_elems(fmt), bb = oracle_block_bytes(fmt);
    if (be == 0 || K <= 0 || K % be != 0) return -1;
    int64_t row_bytes = (K / be) * bb;
    for (int64_t i = 0; i < P; ++i) {
        int64_t m = m_idx[i], n = n_idx[i];
        if (m < 0 || m >= M || n < 0 || n >= N) return -1;
        const uint8_t *row = W + n * row_bytes;
        double acc = 0.0, mag = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = block_value(fmt, row + (k / be) * bb, (int)(k % be)) * (double)x[m * K + k];
            acc += p;
            mag += fabs(p);
        }
        y[i] = acc;
        if (bound) bound[i] = mag;
    }
    return 0;
}
