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

/* ---- float -> block quantizers (packing helpers) ------------------------------
 *
 * The pages quantize weights at load time ("oxinfer" crate page, How it works:
 * quant.rs gives Q8 blocks of 32 weights with one scale and Q4_0 two nibbles
 * per byte with an f16 scale; "wgpu-llm" README, INT8 mode: a quantizer with
 * block size 64) but state no rounding rule.  The reading taken here:
 *
 *   Q8_0, INT8-B64: d = the binary16 value nearest to max|w| / 127 (ties to
 *     even); q = the integer nearest to w / d (ties away from zero), clamped
 *     to -127..127.  A block of zeros, or one whose d rounds to zero, stores
 *     d = +0 and q = 0.
 *   Q4_0: m = the element of largest |w| (the first one when several tie);
 *     d = the binary16 value nearest to m / -8, so that m itself comes back
 *     as d * (0 - 8); q = (integer nearest to w / d, ties away from zero) + 8,
 *     clamped to 0..15.  d = +0 gives q = 8 (value 0).
 *
 * Everything is computed in double: w / d of two floats is correctly rounded
 * there, and that rounding can never move a quotient onto or off a half-way
 * point, so the integer chosen is the one the exact quotient gives.  A
 * non-finite input, or a scale beyond the largest binary16 value (65504),
 * fails the call. */

/* binary16 bits of the value nearest to v (ties to even), written from the
 * format: values k * 2^-24 below 2^-14 (subnormal), k * 2^(e-10) in
 * [2^e, 2^(e+1)).  Returns -1 if v is not finite or rounds past 65504. */
static int double_to_fp16_bits(double v, uint16_t *bits)
{
    if (!isfinite(v)) return -1;
    int sign = signbit(v) ? 1 : 0;
    double a = fabs(v);
    double spacing;
    if (a < ldexp(1.0, -14)) {
        spacing = ldexp(1.0, -24);
    } else {
        int e;
        frexp(a, &e);                      /* a in [2^(e-1), 2^e) */
        spacing = ldexp(1.0, e - 1 - 10);
    }
    double k = a / spacing;                /* exact: spacing is a power of two */
    double kf = floor(k);
    double rest = k - kf;
    if (rest > 0.5 || (rest == 0.5 && fmod(kf, 2.0) == 1.0)) kf += 1.0;
    double r = kf * spacing;               /* exact */
    if (r > 65504.0) return -1;
    uint16_t h;
    if (r == 0.0) {
        h = 0;
    } else if (r < ldexp(1.0, -14)) {
        h = (uint16_t)(r / ldexp(1.0, -24));
    } else {
        int e;
        double f = frexp(r, &e);           /* r = f * 2^e, f in [0.5, 1) */
        int ex = e - 1;                    /* r = (2f) * 2^ex, 2f in [1, 2) */
        int frac = (int)((2.0 * f - 1.0) * 1024.0);
        h = (uint16_t)(((ex + 15) << 10) | frac);
    }
    if (sign) h |= 0x8000;                 /* a negative value that rounds to 0 gives -0 */
    *bits = h;
    return 0;
}

/* the integer nearest to t, ties away from zero (exact for |t| < 2^52) */
static double round_half_away(double t)
{
    double a = fabs(t);
    double f = floor(a);
    if (a - f >= 0.5) f += 1.0;
    return t < 0 ? -f : f;
}

static int quantize_block(int fmt, const float *w, uint8_t *blk)
{
    int be = oracle_block_elems(fmt);
    for (int j = 0; j < be; ++j)
        if (!isfinite(w[j])) return -1;
    uint16_t dbits = 0;
    if (fmt == ORACLE_Q4_0) {
        double m = 0.0;
        for (int j = 0; j < be; ++j)
            if (fabs((double)w[j]) > fabs(m)) m = (double)w[j];
        if (m != 0.0 && double_to_fp16_bits(m / -8.0, &dbits)) return -1;
        if ((dbits & 0x7fff) == 0) dbits = 0;  /* a scale that rounds to zero is stored as +0 */
        double d = oracle_fp16_to_double(dbits);
        blk[0] = (uint8_t)(dbits & 0xff);
        blk[1] = (uint8_t)(dbits >> 8);
        memset(blk + 2, 0, 16);
        for (int j = 0; j < be; ++j) {
            double q = 8.0;
            if (d != 0.0) {
                q = round_half_away((double)w[j] / d) + 8.0;
                if (q < 0.0) q = 0.0;
                if (q > 15.0) q = 15.0;
            }
            int qi = (int)q;
            if (j < 16) blk[2 + j] |= (uint8_t)qi;
            else blk[2 + j - 16] |= (uint8_t)(qi << 4);
        }
        return 0;
    }
    if (fmt == ORACLE_Q8_0 || fmt == ORACLE_I8_B64) {
        double amax = 0.0;
        for (int j = 0; j < be; ++j)
            if (fabs((double)w[j]) > amax) amax = fabs((double)w[j]);
        if (amax != 0.0 && double_to_fp16_bits(amax / 127.0, &dbits)) return -1;
        double d = oracle_fp16_to_double(dbits);  /* amax / 127 >= 0: never -0 */
        blk[0] = (uint8_t)(dbits & 0xff);
        blk[1] = (uint8_t)(dbits >> 8);
        for (int j = 0; j < be; ++j) {
            double q = 0.0;
            if (d != 0.0) {
                q = round_half_away((double)w[j] / d);
                if (q < -127.0) q = -127.0;
                if (q > 127.0) q = 127.0;
            }
            blk[2 + j] = (uint8_t)(int8_t)(int)q;
        }
        return 0;
    }
    return -1;  /* Q6_K has no quantizer here */
}

/* w[N][K] fp32 -> canonical blocks (row-major, blocks along K).  0 on
 * success, -1 on a bad format / shape or an input the reading rejects. */
int oracle_quantize(int fmt, const float *w, uint8_t *canon, int64_t N, int64_t K)
{
    int be = oracle_block_elems(fmt), bb = oracle_block_bytes(fmt);
    if (fmt == ORACLE_Q6_K || be == 0 || N <= 0 || K <= 0 || K % be != 0) return -1;
    for (int64_t n = 0; n < N; ++n)
        for (int64_t b = 0; b < K / be; ++b)
            if (quantize_block(fmt, w + n * K + b * be, canon + (n * (K / be) + b) * bb))
                return -1;
    return 0;
}

/* For the tests: binary16 bits of the value nearest to v, or -1. */
int oracle_double_to_fp16(double v)
{
    uint16_t h;
    return double_to_fp16_bits(v, &h) ? -1 : (int)h;
}

/* ---- the product with x quantized to int8 (activation quantization) ----------
 *
 * The "oxinfer" crate page (How it works) quantizes each matmul's activations
 * so that its decode kernels can run int8 dot products.  It states no rule;
 * the reading taken here is the one its Q8 weights use, with an fp32 scale:
 * per block of 32 consecutive elements of x (along K),
 *     s = max|x| / 127                       (fp32 division)
 *     q = the integer nearest to x / s, ties away from zero, in -127..127
 *                                            (x / s an fp32 division)
 * with s = 0 and q = 0 for a block of zeros.  The product then uses the
 * dequantized activation x~ = s * q:
 *     y[m,n] = sum_k w[n,k] * s_b(k) * q[m,k]      (fp64)
 *     B[m,n] = sum_k |w[n,k] * s_b(k) * q[m,k]|
 * Both rounding decisions are fp32 operations, so any implementation that
 * follows the rule in fp32 picks the same codes. */

/* xq[32], scale of one block of 32 fp32 values (finite). */
static void quantize_x_block(const float *x, int8_t *xq, float *scale)
{
    float amax = 0.0f;
    for (int j = 0; j < 32; ++j) {
        float a = fabsf(x[j]);
        if (a > amax) amax = a;
    }
    volatile float s = amax / 127.0f;   /* an fp32 division, kept in fp32 */
    *scale = s;
    for (int j = 0; j < 32; ++j) {
        if (s == 0.0f) { xq[j] = 0; continue; }
        volatile float t = x[j] / s;      /* an fp32 division */
        float r = roundf(t);              /* ties away from zero */
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        xq[j] = (int8_t)r;
    }
}

/* x[M][K] fp32 -> codes xq[M][K] and scales[M][K/32].  K % 32 == 0. */
int oracle_quantize_x_int8(const float *x, int8_t *xq, float *scales, int64_t M, int64_t K)
{
    if (K <= 0 || K % 32 != 0 || M < 0) return -1;
    for (int64_t m = 0; m < M; ++m)
        for (int64_t b = 0; b < K / 32; ++b)
            quantize_x_block(x + m * K + 32 * b, xq + m * K + 32 * b, scales + m * (K / 32) + b);
    return 0;
}

/* y, bound of the product with x quantized as above. */
int oracle_qmatmul_x_int8(int fmt, const uint8_t *W, const float *x, double *y, double *bound,
                          int64_t N, int64_t K, int64_t M)
{
    int be = oracle_block_elems(fmt), bb = oracle_block_bytes(fmt);
    if (be == 0 || K <= 0 || K % be != 0 || K % 32 != 0 || M < 0) return -1;
    int8_t *xq = (int8_t *)malloc((size_t)(M * K));
    float *sc = (float *)malloc(sizeof(float) * (size_t)(M * (K / 32) + 1));
    double *w = (double *)malloc(sizeof(double) * (size_t)K);
    if (!xq || !sc || !w) { free(xq); free(sc); free(w); return -2; }
    oracle_quantize_x_int8(x, xq, sc, M, K);
    int64_t row_bytes = (K / be) * bb;
    for (int64_t n = 0; n < N; ++n) {
        oracle_dequant_row(fmt, W + n * row_bytes, K, w);
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, mag = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double xt = (double)sc[m * (K / 32) + k / 32] * (double)xq[m * K + k];
                double p = w[k] * xt;
                acc += p;
                mag += fabs(p);
            }
            y[m * N + n] = acc;
            if (bound) bound[m * N + n] = mag;
        }
    }
    free(xq); free(sc); free(w);
    return 0;
}

/* ---- the gated FFN input: h = silu(W_gate x) * (W_up x) ------------------------
 *
 * A decode layer is N x (attention + FFN) ("wgpu-llm" README, Architecture at
 * a Glance); the FFN of the models the pages run (SmolLM2, Qwen2.5,
 * TinyLlama) feeds its down projection with silu(gate) * up, silu(t) =
 * t / (1 + e^-t).  The oracle composes its own products with SiLU written from
 * that definition, in fp64. */
double oracle_silu(double t)
{
    return t / (1.0 + exp(-t));
}

/* h[n], and the parts the tolerance needs: g, u and their bounds. */
int oracle_swiglu(int fmt, const uint8_t *Wg, const uint8_t *Wu, const float *x, double *h,
                  double *g, double *u, double *bg, double *bu, int64_t N, int64_t K)
{
    int rc = oracle_qmatmul(fmt, Wg, x, g, bg, N, K, 1, 1);
    if (rc) return rc;
    rc = oracle_qmatmul(fmt, Wu, x, u, bu, N, K, 1, 1);
    if (rc) return rc;
    for (int64_t n = 0; n < N; ++n) h[n] = oracle_silu(g[n]) * u[n];
    return 0;
}
