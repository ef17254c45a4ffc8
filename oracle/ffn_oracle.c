/*
 * ffn_oracle.c -- TEST INFRASTRUCTURE.  A plain, slow, float64 CPU statement
 * of the pre-norm SwiGLU feed-forward block.  Only the tests, the smoke check
 * and the benchmark's CPU-baseline leg may load this file's library; the
 * product path never does.  It shares no code with the CUDA library.
 *
 * What it computes (no blocking, no fusion, no reordering beyond the
 * definitions; every sum is a plain left-to-right loop in double):
 *
 *   RMSNorm  -- "When to hand-write a GPU kernel on Apple Silicon", Rung 2
 *               (the row reduction: mean of squares over the row, then the
 *               reciprocal square root of mean + eps) and Rung 4 (squares of
 *               upcast values); the gain g is applied per column after the
 *               normalisation, as the block formula states:
 *                   ms_r   = (1/d) * sum_c x[r,c]^2
 *                   n[r,c] = x[r,c] / sqrt(ms_r + eps) * g[c]
 *   SiLU     -- same page, Rung 1: silu(z) = z / (1 + exp(-z)).
 *   SwiGLU   -- same page, Rung 1: h = silu(gate) * up, one value at a time.
 *   Block    -- "Unfusing a Kernel Made It 1.63x Faster", Finding 1 (gate and
 *               up projections, then the activation) and the block formula:
 *                   G[r,f] = sum_c W_gate[f,c] * n[r,c]
 *                   U[r,f] = sum_c W_up[f,c]   * n[r,c]
 *                   h[r,f] = silu(G[r,f]) * U[r,f]
 *                   y[r,j] = sum_f W_down[j,f] * h[r,f]
 *               Weights are [out x in] row-major.  No intermediate rounding.
 *   Q4       -- "Unfusing a Kernel Made It 1.63x Faster", "The finding that
 *               keeps us honest about microbenchmarks" (18-byte blocks: 16
 *               bytes of nibbles, low and high nibbles of the same bytes, plus
 *               a half-precision scale).  w = (u - 8) * s with u the 4-bit
 *               offset-binary value; the layout is documented at
 *               oracle_q4_dequant below.
 *   Row sum of squares -- "Megakernels on Mac: What Fusion Saves and What It Costs", section "Dependencies and
 *               synchronization": after the down projection produces a hidden
 *               vector, the next RMSNorm needs the sum of squares of all its
 *               elements:
 *                   ss[r] = sum_c y[r,c]^2
 *               (oracle_row_sumsq; with the skip connection, y is the next
 *               layer's input).
 *   Q8_0     -- "Unfusing a Kernel Made It 1.63x Faster", "Finding 2: a
 *               quantized KV cache buys nothing while you're
 *               occupancy-bound" (Q8_0, there for the KV cache): blocks of
 *               32 signed 8-bit values with one half-precision scale,
 *               w = q * s; oracle_q8_dequant below.
 *
 * Build: cc -O2 -ffp-contract=off -fPIC -shared ffn_oracle.c -lm -lpthread
 * (no -ffast-math; -ffp-contract=off keeps x86 and Arm results identical).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- scalars */

double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* IEEE binary16 bits -> double, written out from the format's definition:
 * sign (1 bit), exponent (5 bits, bias 15), fraction (10 bits);
 * exponent 0 means subnormal (fraction * 2^-24), exponent 31 inf/nan. */
double oracle_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);
    return sign ? -v : v;
}

/* IEEE-style 8-bit float e4m3 (the "fn" variant: no infinities) decoded to
 * double: sign (1 bit), exponent (4 bits, bias 7), fraction (3 bits);
 * exponent 0 means subnormal (fraction * 2^-9); exponent 15 with fraction 7
 * is NaN (the only non-finite code, so the largest value is 448). */
double oracle_e4m3_to_double(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xF;
    int f = b & 0x7;
    double v;
    if (e == 0)
        v = ldexp((double)f, -9);
    else if (e == 15 && f == 7)
        v = NAN;
    else
        v = ldexp((double)(8 + f), e - 10);
    return sign ? -v : v;
}

/* ----------------------------------------------------------- thread pool */

typedef void (*range_fn)(void *ctx, int64_t lo, int64_t hi);
typedef struct { range_fn fn; void *ctx; int64_t lo, hi; } range_job;

static void *range_thread(void *p) {
    range_job *j = (range_job *)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

/* Run fn over [0, n) split into nthreads contiguous pieces.  The split only
 * decides which thread evaluates an output; each output is computed by the
 * same sequential loop whatever the thread count. */
static void parallel_range(int64_t n, int nthreads, range_fn fn, void *ctx) {
    if (n <= 0) return;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)n;
    if (nthreads == 1) { fn(ctx, 0, n); return; }
    pthread_t tid[256];
    range_job job[256];
    int started[256];
    for (int t = 0; t < nthreads; ++t) {
        job[t].fn = fn; job[t].ctx = ctx;
        job[t].lo = n * t / nthreads; job[t].hi = n * (t + 1) / nthreads;
        started[t] = pthread_create(&tid[t], NULL, range_thread, &job[t]) == 0;
        if (!started[t]) range_thread(&job[t]);
    }
    for (int t = 0; t < nthreads; ++t)
        if (started[t]) pthread_join(tid[t], NULL);
}

/* --------------------------------------------------------------- RMSNorm */

typedef struct { const double *x, *g; double *n; int64_t d; double eps; } norm_ctx;

static void norm_rows(void *p, int64_t lo, int64_t hi) {
    norm_ctx *c = (norm_ctx *)p;
    for (int64_t r = lo; r < hi; ++r) {
        const double *xr = c->x + r * c->d;
        double *nr = c->n + r * c->d;
        double ss = 0.0;
        for (int64_t k = 0; k < c->d; ++k) ss += xr[k] * xr[k];
        double ms = ss / (double)c->d;
        double root = sqrt(ms + c->eps);
        for (int64_t k = 0; k < c->d; ++k) nr[k] = xr[k] / root * c->g[k];
    }
}

void oracle_rmsnorm(const double *x, const double *g, double *n, int64_t rows,
                    int64_t d, double eps, int nthreads) {
    norm_ctx c = {x, g, n, d, eps};
    parallel_range(rows, nthreads, norm_rows, &c);
}

/* ss[r] = sum over c of y[r,c]^2, a left-to-right sum per row. */
void oracle_row_sumsq(const double *y, double *ss, int64_t rows, int64_t d) {
    for (int64_t r = 0; r < rows; ++r) {
        const double *yr = y + r * d;
        double acc = 0.0;
        for (int64_t c = 0; c < d; ++c) acc += yr[c] * yr[c];
        ss[r] = acc;
    }
}

/* ---------------------------------------------------------------- SwiGLU */

typedef struct { const double *gate, *up; double *h; } swiglu_ctx;

static void swiglu_range(void *p, int64_t lo, int64_t hi) {
    swiglu_ctx *c = (swiglu_ctx *)p;
    for (int64_t i = lo; i < hi; ++i) c->h[i] = oracle_silu(c->gate[i]) * c->up[i];
}

void oracle_swiglu(const double *gate, const double *up, double *h, int64_t count,
                   int nthreads) {
    swiglu_ctx c = {gate, up, h};
    parallel_range(count, nthreads, swiglu_range, &c);
}

/* ------------------------------------------------------------ FFN block */

typedef struct {
    const double *n, *w_gate, *w_up, *w_down;
    double *h, *y;
    int64_t d, ffn;
} block_ctx;

/* h[r,f] for flat index i = r*ffn + f */
static void block_hidden(void *p, int64_t lo, int64_t hi) {
    block_ctx *c = (block_ctx *)p;
    for (int64_t i = lo; i < hi; ++i) {
        int64_t r = i / c->ffn, f = i % c->ffn;
        const double *nr = c->n + r * c->d;
        const double *wg = c->w_gate + f * c->d;
        const double *wu = c->w_up + f * c->d;
        double G = 0.0, U = 0.0;
        for (int64_t k = 0; k < c->d; ++k) G += wg[k] * nr[k];
        for (int64_t k = 0; k < c->d; ++k) U += wu[k] * nr[k];
        c->h[i] = oracle_silu(G) * U;
    }
}

/* y[r,j] for flat index i = r*d + j */
static void block_out(void *p, int64_t lo, int64_t hi) {
    block_ctx *c = (block_ctx *)p;
    for (int64_t i = lo; i < hi; ++i) {
        int64_t r = i / c->d, j = i % c->d;
        const double *hr = c->h + r * c->ffn;
        const double *wd = c->w_down + j * c->ffn;
        double s = 0.0;
        for (int64_t f = 0; f < c->ffn; ++f) s += wd[f] * hr[f];
        c->y[i] = s;
    }
}

/* y = W_down (silu(W_gate n) * (W_up n)),  n = RMSNorm(x; g, eps).
 * x [rows x d], g [d], w_gate/w_up [ffn x d], w_down [d x ffn], y [rows x d].
 * Returns 0, or -1 if scratch memory cannot be allocated. */
int oracle_ffn_block(const double *x, const double *g, const double *w_gate,
                     const double *w_up, const double *w_down, double *y,
                     int64_t rows, int64_t d, int64_t ffn, double eps, int nthreads) {
    double *n = (double *)malloc(sizeof(double) * (size_t)(rows * d > 0 ? rows * d : 1));
    double *h = (double *)malloc(sizeof(double) * (size_t)(rows * ffn > 0 ? rows * ffn : 1));
    if (!n || !h) { free(n); free(h); return -1; }
    oracle_rmsnorm(x, g, n, rows, d, eps, nthreads);
    block_ctx c = {n, w_gate, w_up, w_down, h, y, d, ffn};
    parallel_range(rows * ffn, nthreads, block_hidden, &c);
    parallel_range(rows * d, nthreads, block_out, &c);
    free(n);
    free(h);
    return 0;
}

/* ------------------------------------------------------------------- Q4 */

/* Dequantise Q4 weights from the device layout into double w[out x in].
 *
 * Canonical block (32 weights, one fp16 scale s): weight j is stored as the
 * offset-binary nibble u_j = q_j + 8; canonical byte i (0..15) holds u_i in
 * its low nibble and u_(i+16) in its high nibble; w_j = (u_j - 8) * s.
 *
 * Device layout: blocks are taken four at a time along the input dimension
 * (a group of 128 weights, 64 bytes); byte 16*t + 4*b + e of a group is
 * canonical byte 4*t + e of block b of that group.  A weight row holds
 * ceil(in/128) groups (in/2 bytes when in is a multiple of 128); blocks of
 * a last, partial group past in/32 are padding and are not read.  Scales
 * [out][4*ceil(in/128)]: scales[o][blk] holds the fp16 bits of block blk's
 * scale. */
void oracle_q4_dequant(const uint8_t *qs, const uint16_t *scales, double *w,
                       int64_t out, int64_t in) {
    int64_t nblk = in / 32;
    int64_t ngrp = (in + 127) / 128;
    for (int64_t o = 0; o < out; ++o) {
        const uint8_t *row = qs + o * ngrp * 64;
        for (int64_t blk = 0; blk < nblk; ++blk) {
            double s = oracle_half_to_double(scales[o * ngrp * 4 + blk]);
            int64_t group = blk / 4;
            int b = (int)(blk % 4);
            const uint8_t *gp = row + group * 64;
            for (int j = 0; j < 32; ++j) {
                int i = j % 16;                  /* canonical byte */
                int t = i / 4, e = i % 4;
                uint8_t byte = gp[16 * t + 4 * b + e];
                int u = (j < 16) ? (byte & 0x0F) : (byte >> 4);
                w[o * in + blk * 32 + j] = (double)(u - 8) * s;
            }
        }
    }
}

/* ----------------------------------------------------------------- Q8_0 */

/* Dequantise Q8_0 weights into double w[out x in].  Blocks of 32 weights run
 * along the input dimension, each with one fp16 scale; q[o][i] is a signed
 * byte (two's complement, -128..127) and w[o][i] = q[o][i] * s[o][i / 32].
 * The layout keeps the bytes in natural order, [out x in], and the scales in
 * their own array [out x in/32] (a block's 34 bytes, split in two). */
void oracle_q8_dequant(const int8_t *q, const uint16_t *scales, double *w, int64_t out, int64_t in) {
    int64_t nblk = in / 32;
    for (int64_t o = 0; o < out; ++o)
        for (int64_t i = 0; i < in; ++i)
            w[o * in + i] = (double)q[o * in + i] * oracle_half_to_double(scales[o * nblk + i / 32]);
}

/* ------------------------------------------------------------------ fp8 */

/* Dequantise fp8 weights: codes[o][i] is an e4m3 byte, scales[o] the row's
 * float scale; w[o][i] = e4m3(codes[o][i]) * scales[o], exact in double. */
void oracle_fp8_dequant(const uint8_t *codes, const float *scales, double *w, int64_t out, int64_t in) {
    for (int64_t o = 0; o < out; ++o) {
        const double s = (double)scales[o];
        for (int64_t i = 0; i < in; ++i) w[o * in + i] = oracle_e4m3_to_double(codes[o * in + i]) * s;
    }
}
