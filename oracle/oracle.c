/*
 * Plain fp64 CPU oracle for the dense video-token attention path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no code, header or constant with the CUDA path.
 *
 * Every function is the plain definition written out, in double precision,
 * with no tiling, fusion or reordering:
 *
 *   oracle_attn_rows      softmax(q K^T * scale) V for chosen query rows of one
 *                         head, plus log-sum-exp.  Full, unmasked attention over
 *                         the packed sequence: "FreeVideo: a 66 GB video
 *                         transformer on an 8 GB card", sections "What MiniMax
 *                         H3 is, briefly" (56 heads of 128) and "Why it does not
 *                         fit: the arithmetic" (dense scores, streamed by
 *                         flash-style kernels); "FastH3 Preview v1", section
 *                         "Lever two: VSA-H3 ..." (one joint bidirectional
 *                         attention over the packed sequence).
 *   oracle_modulate       y = LN(x) * (1 + scale[step]) + shift[step], LN
 *                         without learned affine, biased variance: "FreeVideo",
 *                         section "Cut one: 26 GB of AdaLN weights become 0.22 GB
 *                         of tables" (shift, scale and gate per step, read from
 *                         a stored table).
 *   oracle_gated_residual out = x + gate[step] * a, then rounded to bfloat16
 *                         (same section: the gate of the attention branch).
 *   oracle_attn_rows_window  the softmax branch of Video DeltaNet: the same
 *                         attention over the keys of a local window of latent
 *                         frames plus the first and last frame ("FreeVideo",
 *                         section "Where Video DeltaNet comes in").
 *
 * Inputs are bfloat16 bit patterns (uint16) and float32 tables; both convert
 * exactly to double.  Work is split over rows with POSIX threads; each row is
 * computed exactly as written, independently of the split.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bfloat16 bits -> double (exact: a bfloat16 is the top half of a float). */
static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> nearest bfloat16 value, ties to even, returned as a double.
 * bfloat16 keeps 8 significant bits and float32's exponent range
 * (normal 2^-126 .. (2 - 2^-7) 2^127, subnormal spacing 2^-133). */
double oracle_round_bf16(double x) {
    if (isnan(x) || isinf(x) || x == 0.0) return x;
    int e;
    frexp(x, &e);                     /* x = f 2^e, 0.5 <= |f| < 1 */
    int q = e - 8;                    /* spacing of 8-bit significands at this binade */
    if (q < -133) q = -133;           /* subnormal range: fixed spacing */
    double r = nearbyint(ldexp(x, -q));   /* default rounding mode: ties to even */
    double y = ldexp(r, q);
    const double maxv = ldexp(255.0, 120);  /* (2 - 2^-7) * 2^127 */
    if (fabs(y) > maxv) y = copysign(INFINITY, x);
    return y;
}

uint16_t oracle_bf16_bits(double x) {
    float f = (float)oracle_round_bf16(x);  /* exact: the value is a bfloat16 */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* attention                                                                 */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint16_t *Q;       /* [N, ld] bf16, head columns [h*D, h*D+D) */
    const double *Kd, *Vd;   /* this head's K and V as double, [N, D] */
    int64_t N, ld;
    int D, h;
    double scale;
    const int64_t *rows;
    int64_t r_begin, r_end;
    double *O;               /* [nrows, D] */
    double *lse;             /* [nrows] */
} attn_job;

static void *attn_worker(void *arg) {
    attn_job *j = (attn_job *)arg;
    const int64_t N = j->N;
    const int D = j->D;
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
    double *q = (double *)malloc(sizeof(double) * (size_t)D);
    for (int64_t r = j->r_begin; r < j->r_end; ++r) {
        const int64_t i = j->rows[r];
        for (int c = 0; c < D; ++c) q[c] = bf16_to_double(j->Q[i * j->ld + (int64_t)j->h * D + c]);
        /* s_ij = scale * q_i . k_j for every key j (no mask) */
        for (int64_t t = 0; t < N; ++t) {
            const double *k = j->Kd + t * D;
            double dot = 0.0;
            for (int c = 0; c < D; ++c) dot += q[c] * k[c];
            s[t] = j->scale * dot;
        }
        /* m = max_j s_ij */
        double m = -INFINITY;
        for (int64_t t = 0; t < N; ++t) if (s[t] > m) m = s[t];
        /* e_j = exp(s_ij - m), l = sum_j e_j */
        double l = 0.0;
        for (int64_t t = 0; t < N; ++t) { s[t] = exp(s[t] - m); l += s[t]; }
        /* o_i = sum_j e_j v_j / l */
        double *o = j->O + r * D;
        for (int c = 0; c < D; ++c) o[c] = 0.0;
        for (int64_t t = 0; t < N; ++t) {
            const double *v = j->Vd + t * D;
            for (int c = 0; c < D; ++c) o[c] += s[t] * v[c];
        }
        for (int c = 0; c < D; ++c) o[c] /= l;
        j->lse[r] = m + log(l);
    }
    free(q);
    free(s);
    return NULL;
}

static int clamp_threads(int nthreads, int64_t work) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > work) nthreads = (int)(work > 0 ? work : 1);
    return nthreads;
}

/*
 * Attention output of head h for query rows rows[0..nrows).
 * Q, K, V: bf16 [N, ld] row-major (ld = H*D), head h in columns [h*D, h*D+D).
 * O: double [nrows, D]; lse: double [nrows] (natural log).
 * Returns 0, or -1 on bad arguments / allocation failure.
 */
int oracle_attn_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                     int64_t N, int64_t ld, int D, int h, double scale,
                     const int64_t *rows, int64_t nrows,
                     double *O, double *lse, int nthreads) {
    if (!Q || !K || !V || !rows || !O || !lse || N < 1 || D < 1 || h < 0 ||
        ld < (int64_t)(h + 1) * D || nrows < 0)
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -1;
    if (nrows == 0) return 0;
    double *Kd = (double *)malloc(sizeof(double) * (size_t)N * (size_t)D);
    double *Vd = (double *)malloc(sizeof(double) * (size_t)N * (size_t)D);
    if (!Kd || !Vd) { free(Kd); free(Vd); return -1; }
    for (int64_t t = 0; t < N; ++t)
        for (int c = 0; c < D; ++c) {
            Kd[t * D + c] = bf16_to_double(K[t * ld + (int64_t)h * D + c]);
            Vd[t * D + c] = bf16_to_double(V[t * ld + (int64_t)h * D + c]);
        }
    nthreads = clamp_threads(nthreads, nrows);
    pthread_t tid[256];
    attn_job job[256];
    for (int w = 0; w < nthreads; ++w) {
        attn_job *j = &job[w];
        j->Q = Q; j->Kd = Kd; j->Vd = Vd; j->N = N; j->ld = ld; j->D = D; j->h = h;
        j->scale = scale; j->rows = rows; j->O = O; j->lse = lse;
        j->r_begin = nrows * w / nthreads;
        j->r_end = nrows * (w + 1) / nthreads;
        pthread_create(&tid[w], NULL, attn_worker, j);
    }
    for (int w = 0; w < nthreads; ++w) pthread_join(tid[w], NULL);
    free(Kd);
    free(Vd);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* windowed attention (Video DeltaNet softmax branch)                        */
/* ------------------------------------------------------------------------ */
/*
 * Which keys query i may see ("FreeVideo", section "Where Video DeltaNet
 * comes in"): tokens are grouped into latent frames of T tokens and frames
 * into chunks of C frames (one VAE chunk); a query sees every key whose chunk
 * is within W chunks of its own (W = 1: itself and its two neighbours, a
 * 15-frame window), plus every key in the first and the last latent frame;
 * queries in the first and the last latent frame see every key.
 */
int oracle_window_allowed(int64_t i, int64_t j, int64_t N, int64_t T, int64_t C, int64_t W) {
    const int64_t frames = N / T;
    const int64_t fi = i / T, fj = j / T;
    if (fi == 0 || fi == frames - 1) return 1;
    if (fj == 0 || fj == frames - 1) return 1;
    int64_t d = fi / C - fj / C;
    if (d < 0) d = -d;
    return d <= W;
}

typedef struct {
    attn_job a;
    int64_t T, C, W;
} win_job;

static void *win_worker(void *arg) {
    win_job *w = (win_job *)arg;
    attn_job *j = &w->a;
    const int64_t N = j->N;
    const int D = j->D;
    double *s = (double *)malloc(sizeof(double) * (size_t)N);
    double *q = (double *)malloc(sizeof(double) * (size_t)D);
    for (int64_t r = j->r_begin; r < j->r_end; ++r) {
        const int64_t i = j->rows[r];
        for (int c = 0; c < D; ++c) q[c] = bf16_to_double(j->Q[i * j->ld + (int64_t)j->h * D + c]);
        /* scores of the allowed keys; -inf marks a key the query may not see */
        for (int64_t t = 0; t < N; ++t) {
            if (!oracle_window_allowed(i, t, N, w->T, w->C, w->W)) { s[t] = -INFINITY; continue; }
            const double *k = j->Kd + t * D;
            double dot = 0.0;
            for (int c = 0; c < D; ++c) dot += q[c] * k[c];
            s[t] = j->scale * dot;
        }
        double m = -INFINITY;
        for (int64_t t = 0; t < N; ++t) if (s[t] > m) m = s[t];
        double l = 0.0;
        for (int64_t t = 0; t < N; ++t) { s[t] = (s[t] == -INFINITY) ? 0.0 : exp(s[t] - m); l += s[t]; }
        double *o = j->O + r * D;
        for (int c = 0; c < D; ++c) o[c] = 0.0;
        for (int64_t t = 0; t < N; ++t) {
            if (s[t] == 0.0) continue;
            const double *v = j->Vd + t * D;
            for (int c = 0; c < D; ++c) o[c] += s[t] * v[c];
        }
        for (int c = 0; c < D; ++c) o[c] /= l;
        j->lse[r] = m + log(l);
    }
    free(q);
    free(s);
    return NULL;
}

/*
 * Windowed attention of head h for query rows rows[0..nrows): the same as
 * oracle_attn_rows over the keys oracle_window_allowed admits.  N must be a
 * multiple of T.
 */
int oracle_attn_rows_window(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                            int64_t N, int64_t ld, int D, int h, double scale,
                            int64_t T, int64_t C, int64_t W,
                            const int64_t *rows, int64_t nrows,
                            double *O, double *lse, int nthreads) {
    if (!Q || !K || !V || !rows || !O || !lse || N < 1 || D < 1 || h < 0 ||
        ld < (int64_t)(h + 1) * D || nrows < 0 || T < 1 || N % T != 0 || C < 1 || W < 0)
        return -1;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -1;
    if (nrows == 0) return 0;
    double *Kd = (double *)malloc(sizeof(double) * (size_t)N * (size_t)D);
    double *Vd = (double *)malloc(sizeof(double) * (size_t)N * (size_t)D);
    if (!Kd || !Vd) { free(Kd); free(Vd); return -1; }
    for (int64_t t = 0; t < N; ++t)
        for (int c = 0; c < D; ++c) {
            Kd[t * D + c] = bf16_to_double(K[t * ld + (int64_t)h * D + c]);
            Vd[t * D + c] = bf16_to_double(V[t * ld + (int64_t)h * D + c]);
        }
    nthreads = clamp_threads(nthreads, nrows);
    pthread_t tid[256];
    win_job job[256];
    for (int w = 0; w < nthreads; ++w) {
        attn_job *j = &job[w].a;
        j->Q = Q; j->Kd = Kd; j->Vd = Vd; j->N = N; j->ld = ld; j->D = D; j->h = h;
        j->scale = scale; j->rows = rows; j->O = O; j->lse = lse;
        j->r_begin = nrows * w / nthreads;
        j->r_end = nrows * (w + 1) / nthreads;
        job[w].T = T; job[w].C = C; job[w].W = W;
        pthread_create(&tid[w], NULL, win_worker, &job[w]);
    }
    for (int w = 0; w < nthreads; ++w) pthread_join(tid[w], NULL);
    free(Kd);
    free(Vd);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* AdaLN modulate and gated residual                                         */
/* ------------------------------------------------------------------------ */
typedef struct {
    const uint16_t *x, *a;
    const float *t0, *t1;    /* modulate: shift row, scale row; residual: gate row */
    int64_t C;
    double eps;
    const int64_t *rows;
    int64_t r_begin, r_end;
    double *y;               /* [nrows, C] */
    uint16_t *ybits;         /* residual only: [nrows, C] bf16 bits */
} row_job;

static void *modulate_worker(void *arg) {
    row_job *j = (row_job *)arg;
    const int64_t C = j->C;
    for (int64_t r = j->r_begin; r < j->r_end; ++r) {
        const uint16_t *x = j->x + j->rows[r] * C;
        /* mean, then biased variance of the deviations (two passes) */
        double mu = 0.0;
        for (int64_t c = 0; c < C; ++c) mu += bf16_to_double(x[c]);
        mu /= (double)C;
        double var = 0.0;
        for (int64_t c = 0; c < C; ++c) { double d = bf16_to_double(x[c]) - mu; var += d * d; }
        var /= (double)C;
        const double inv = 1.0 / sqrt(var + j->eps);
        double *y = j->y + r * C;
        for (int64_t c = 0; c < C; ++c) {
            double n = (bf16_to_double(x[c]) - mu) * inv;
            y[c] = n * (1.0 + (double)j->t1[c]) + (double)j->t0[c];
        }
    }
    return NULL;
}

static void *residual_worker(void *arg) {
    row_job *j = (row_job *)arg;
    const int64_t C = j->C;
    for (int64_t r = j->r_begin; r < j->r_end; ++r) {
        const uint16_t *x = j->x + j->rows[r] * C;
        const uint16_t *a = j->a + j->rows[r] * C;
        for (int64_t c = 0; c < C; ++c) {
            double v = bf16_to_double(x[c]) + (double)j->t0[c] * bf16_to_double(a[c]);
            j->y[r * C + c] = v;
            j->ybits[r * C + c] = oracle_bf16_bits(v);
        }
    }
    return NULL;
}

static int run_rows(void *(*fn)(void *), row_job base, int64_t nrows, int nthreads) {
    nthreads = clamp_threads(nthreads, nrows);
    pthread_t tid[256];
    row_job job[256];
    for (int w = 0; w < nthreads; ++w) {
        job[w] = base;
        job[w].r_begin = nrows * w / nthreads;
        job[w].r_end = nrows * (w + 1) / nthreads;
        pthread_create(&tid[w], NULL, fn, &job[w]);
    }
    for (int w = 0; w < nthreads; ++w) pthread_join(tid[w], NULL);
    return 0;
}

/*
 * y[r, :] = LN(x[rows[r], :]) * (1 + scale_row) + shift_row, in double.
 * x: bf16 [*, C]; shift_row, scale_row: float [C] (the table row of the step).
 */
int oracle_modulate(const uint16_t *x, int64_t C, const float *shift_row, const float *scale_row,
                    double eps, const int64_t *rows, int64_t nrows, double *y, int nthreads) {
    if (!x || !shift_row || !scale_row || !rows || !y || C < 1 || nrows < 0 || !(eps >= 0.0))
        return -1;
    if (nrows == 0) return 0;
    row_job b;
    memset(&b, 0, sizeof b);
    b.x = x; b.t0 = shift_row; b.t1 = scale_row; b.C = C; b.eps = eps; b.rows = rows; b.y = y;
    return run_rows(modulate_worker, b, nrows, nthreads);
}

/*
 * y[r, :] = x[rows[r], :] + gate_row * a[rows[r], :] in double, and ybits the
 * same values rounded to bfloat16 (ties to even).
 */
int oracle_gated_residual(const uint16_t *x, const uint16_t *a, int64_t C, const float *gate_row,
                          const int64_t *rows, int64_t nrows, double *y, uint16_t *ybits,
                          int nthreads) {
    if (!x || !a || !gate_row || !rows || !y || !ybits || C < 1 || nrows < 0) return -1;
    if (nrows == 0) return 0;
    row_job b;
    memset(&b, 0, sizeof b);
    b.x = x; b.a = a; b.t0 = gate_row; b.C = C; b.rows = rows; b.y = y; b.ybits = ybits;
    return run_rows(residual_worker, b, nrows, nthreads);
}
