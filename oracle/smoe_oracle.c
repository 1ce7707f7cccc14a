/*
 * smoe_oracle.c -- plain, slow, f64 CPU oracle for the group-quantized
 * routed-expert FFN and the dense bf16 matvec.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file or the library built from it: only the tests, the smoke
 * check and the benchmark's CPU-baseline leg use it.  It shares no code,
 * header, table or constant with the CUDA library.
 *
 * Source of every definition: the S-MoE documentation page
 * "Metal Compute Kernels":
 *   - section "Fused FFN Kernels -- One Simdgroup Per Output Row":
 *       hidden[i] = SiLU(gate_proj . x)[i] * (up_proj . x)[i]
 *       out[j]    = (down_proj . hidden)[j]
 *       w = (code - Z) * (1/Z) * s, with Z = 7.5 for Q4 and Z = 1.5 for Q2,
 *       one scale s per (row, group of input columns).
 *   - section "Layout assumptions the kernels rely on": codes are packed
 *       along a row; cols % 32 (Q4) / % 64 (Q2); group size 64.
 *   - section "Coalesced Dense Matvec -- the Same Contract for bf16":
 *       y = W x with bf16 weights, f32 input and output.
 *   - section "Token-Batch Fused FFN": the same FFN applied to every row of
 *       a [batch x d_model] input.
 *
 * Readings where the page is silent (each one is listed with its reason in
 * the design notes):
 *   - Q4 packing: byte j of a row holds column 2j in its low nibble and
 *     column 2j+1 in its high nibble.
 *   - Q2 packing: byte j holds columns 4j..4j+3, the first column in the
 *     lowest two bits.
 *   - scales are f32, row-major [rows][cols/group].
 *   - SiLU(v) = v / (1 + exp(-v)).
 *
 * The oracle deliberately does NOT use the method's folded form
 * s*((sum code*x)/Z - sum x): it dequantises every single weight to f64 and
 * dots it with x, which is the plain definition the fold must reproduce.
 * Every product also adds |w*x| into a second sum, which the tests use for
 * the per-element tolerance 1e-4 * sum|w*x| + 1e-6.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAX_THREADS 256

static int g_threads = 1;

/* Number of host threads the row loops below are split over (>= 1). */
int oracle_set_threads(int n)
{
    if (n < 1) n = 1;
    if (n > ORACLE_MAX_THREADS) n = ORACLE_MAX_THREADS;
    g_threads = n;
    return g_threads;
}

int oracle_get_threads(void) { return g_threads; }

/* Z, the code offset: 7.5 at Q4, 1.5 at Q2 ("Fused FFN Kernels"). */
static double zero_point(int bits) { return bits == 4 ? 7.5 : 1.5; }

/* The code of column k of one packed row (reading of the packing above). */
int oracle_code_at(const uint8_t *row, int bits, long k)
{
    if (bits == 4) {
        uint8_t b = row[k / 2];
        return (k % 2 == 0) ? (b & 0x0F) : (b >> 4);
    }
    uint8_t b = row[k / 4];
    return (b >> (2 * (k % 4))) & 0x03;
}

/* Unpacks n codes of a packed stream, one code per output byte. */
int oracle_unpack(const uint8_t *packed, int bits, long n, uint8_t *codes)
{
    if (bits != 4 && bits != 2) return -1;
    for (long k = 0; k < n; ++k) codes[k] = (uint8_t)oracle_code_at(packed, bits, k);
    return 0;
}

/* w = (code - Z) * (1/Z) * s, in f64. */
double oracle_dequant(int code, int bits, double scale)
{
    double z = zero_point(bits);
    return (code - z) / z * scale;
}

/* SiLU(v) = v * sigmoid(v) = v / (1 + e^-v). */
double oracle_silu(double v) { return v / (1.0 + exp(-v)); }

/* bf16 bit pattern -> the f32 it denotes (upper half of an f32) -> f64. */
double oracle_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ------------------------------------------------------------------------ */
/* Row-parallel driver: the same per-row function, rows split over threads. */

typedef void (*row_fn)(void *ctx, long r);

struct row_task {
    row_fn fn;
    void *ctx;
    long r0, r1;
};

static void *row_task_main(void *arg)
{
    struct row_task *t = (struct row_task *)arg;
    for (long r = t->r0; r < t->r1; ++r) t->fn(t->ctx, r);
    return NULL;
}

static void for_rows(row_fn fn, void *ctx, long r0, long r1)
{
    long n = r1 - r0;
    int nt = g_threads;
    if (nt > n) nt = (int)(n > 0 ? n : 1);
    if (nt <= 1) {
        for (long r = r0; r < r1; ++r) fn(ctx, r);
        return;
    }
    pthread_t th[ORACLE_MAX_THREADS];
    struct row_task task[ORACLE_MAX_THREADS];
    int started[ORACLE_MAX_THREADS];
    for (int i = 0; i < nt; ++i) {
        task[i].fn = fn;
        task[i].ctx = ctx;
        task[i].r0 = r0 + n * i / nt;
        task[i].r1 = r0 + n * (i + 1) / nt;
        started[i] = pthread_create(&th[i], NULL, row_task_main, &task[i]) == 0;
        if (!started[i]) row_task_main(&task[i]);
    }
    for (int i = 0; i < nt; ++i)
        if (started[i]) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------ */
/* Group-quantized matvec: y[r] = sum_k w[r][k] * x[k].                       */

struct qgemv_ctx {
    int bits;
    const uint8_t *codes;
    const float *scales;
    long cols, group, row0;
    const double *x;
    double *y, *absdot;
};

static void qgemv_row(void *p, long r)
{
    const struct qgemv_ctx *c = (const struct qgemv_ctx *)p;
    long row_bytes = c->cols * c->bits / 8;
    long ngroups = c->cols / c->group;
    const uint8_t *crow = c->codes + r * row_bytes;
    const float *srow = c->scales + r * ngroups;
    double acc = 0.0, mag = 0.0;
    for (long k = 0; k < c->cols; ++k) {
        double w = oracle_dequant(oracle_code_at(crow, c->bits, k), c->bits,
                                  (double)srow[k / c->group]);
        double t = w * c->x[k];
        acc += t;
        mag += fabs(t);
    }
    c->y[r - c->row0] = acc;
    if (c->absdot) c->absdot[r - c->row0] = mag;
}

static int q_args_ok(int bits, long rows, long cols, long group)
{
    if (bits != 4 && bits != 2) return 0;
    if (rows < 0 || cols < 0 || group <= 0) return 0;
    if (cols % group != 0) return 0;
    if ((cols * bits) % 8 != 0) return 0;
    return 1;
}

/*
 * Rows [row0, row0 + nrows) of y = W x for a packed [rows x cols] matrix.
 * y and absdot (may be NULL) receive nrows values.  Returns 0, or -1 on bad
 * arguments.
 */
int oracle_qgemv(int bits, const uint8_t *codes, const float *scales, long rows,
                 long cols, long group, const double *x, long row0, long nrows,
                 double *y, double *absdot)
{
    if (!q_args_ok(bits, rows, cols, group)) return -1;
    if (row0 < 0 || nrows < 0 || row0 + nrows > rows) return -1;
    struct qgemv_ctx c = {bits, codes, scales, cols, group, row0, x, y, absdot};
    for_rows(qgemv_row, &c, row0, row0 + nrows);
    return 0;
}

/*
 * Fused gate/up for hidden rows [row0, row0 + nrows):
 *   g = gate . x, u = up . x, hidden = SiLU(g) * u.
 * g, u, g_abs, u_abs may be NULL.
 */
int oracle_gate_up(int bits, const uint8_t *gate_codes, const float *gate_scales,
                   const uint8_t *up_codes, const float *up_scales, long d_ff,
                   long d_model, long group, const double *x, long row0, long nrows,
                   double *hidden, double *g, double *u, double *g_abs, double *u_abs)
{
    if (!q_args_ok(bits, d_ff, d_model, group)) return -1;
    if (row0 < 0 || nrows < 0 || row0 + nrows > d_ff) return -1;
    double *gv = (double *)malloc(sizeof(double) * (size_t)(nrows > 0 ? nrows : 1));
    double *uv = (double *)malloc(sizeof(double) * (size_t)(nrows > 0 ? nrows : 1));
    if (!gv || !uv) {
        free(gv);
        free(uv);
        return -1;
    }
    oracle_qgemv(bits, gate_codes, gate_scales, d_ff, d_model, group, x, row0, nrows, gv, g_abs);
    oracle_qgemv(bits, up_codes, up_scales, d_ff, d_model, group, x, row0, nrows, uv, u_abs);
    for (long i = 0; i < nrows; ++i) {
        hidden[i] = oracle_silu(gv[i]) * uv[i];
        if (g) g[i] = gv[i];
        if (u) u[i] = uv[i];
    }
    free(gv);
    free(uv);
    return 0;
}

/*
 * One expert, one token: hidden = SiLU(gate.x) * (up.x) over all d_ff rows,
 * then out = down . hidden over all d_model rows (down is [d_model x d_ff],
 * grouped along d_ff).  hidden (d_ff values), out and out_abs (d_model values)
 * are written; out_abs may be NULL.
 */
int oracle_ffn(int bits, const uint8_t *gate_codes, const float *gate_scales,
               const uint8_t *up_codes, const float *up_scales,
               const uint8_t *down_codes, const float *down_scales, long d_model,
               long d_ff, long group, const double *x, double *hidden, double *out,
               double *out_abs)
{
    if (!q_args_ok(bits, d_model, d_ff, group)) return -1;
    int rc = oracle_gate_up(bits, gate_codes, gate_scales, up_codes, up_scales, d_ff,
                            d_model, group, x, 0, d_ff, hidden, NULL, NULL, NULL, NULL);
    if (rc) return rc;
    return oracle_qgemv(bits, down_codes, down_scales, d_model, d_ff, group, hidden, 0,
                        d_model, out, out_abs);
}

/*
 * Token batch: the one-token FFN above applied to rows [t0, t0 + nt) of
 * X [T x d_model].  hidden receives nt*d_ff values, Y and Y_abs nt*d_model.
 */
int oracle_ffn_batch(int bits, const uint8_t *gate_codes, const float *gate_scales,
                     const uint8_t *up_codes, const float *up_scales,
                     const uint8_t *down_codes, const float *down_scales, long T,
                     long d_model, long d_ff, long group, const double *X, long t0,
                     long nt, double *hidden, double *Y, double *Y_abs)
{
    if (T < 0 || t0 < 0 || nt < 0 || t0 + nt > T) return -1;
    for (long t = 0; t < nt; ++t) {
        int rc = oracle_ffn(bits, gate_codes, gate_scales, up_codes, up_scales, down_codes,
                            down_scales, d_model, d_ff, group, X + (t0 + t) * d_model,
                            hidden + t * d_ff, Y + t * d_model,
                            Y_abs ? Y_abs + t * d_model : NULL);
        if (rc) return rc;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Dense bf16 matvec: y[r] = sum_k bf16(W[r][k]) * x[k].                      */

struct bf16_ctx {
    const uint16_t *w;
    long cols, row0;
    const double *x;
    double *y, *absdot;
};

static void bf16_row(void *p, long r)
{
    const struct bf16_ctx *c = (const struct bf16_ctx *)p;
    const uint16_t *wrow = c->w + r * c->cols;
    double acc = 0.0, mag = 0.0;
    for (long k = 0; k < c->cols; ++k) {
        double t = oracle_bf16_value(wrow[k]) * c->x[k];
        acc += t;
        mag += fabs(t);
    }
    c->y[r - c->row0] = acc;
    if (c->absdot) c->absdot[r - c->row0] = mag;
}

/* Rows [row0, row0 + nrows) of y = W x, W given as [rows x cols] bf16 bits. */
int oracle_matvec_bf16(const uint16_t *w, long rows, long cols, const double *x,
                       long row0, long nrows, double *y, double *absdot)
{
    if (rows < 0 || cols < 0 || row0 < 0 || nrows < 0 || row0 + nrows > rows) return -1;
    struct bf16_ctx c = {w, cols, row0, x, y, absdot};
    for_rows(bf16_row, &c, row0, row0 + nrows);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Routing and combine.  The pages run the exact-routing gate matvec (n_experts
 * x d_model) on the host and describe neither the selection nor the
 * weighting; the readings taken here:
 *   logits = G x with bf16 G (the matvec above);
 *   the k experts with the largest logits, in descending logit order, ties
 *     to the lower expert index, NaN below every number;
 *   their weights: exp(l_i - l_max) / sum over the k selected of
 *     exp(l_j - l_max) (a softmax over all experts renormalised over the
 *     selected k gives the same values);
 *   combine: out[j] = sum over the k selected, in selection order, of
 *     w_i * y_i[j]. */

/* 1 if (va, ia) ranks before (vb, ib). */
static int ranks_before(double va, long ia, double vb, long ib)
{
    const int na = isnan(va), nb = isnan(vb);
    if (na != nb) return nb;          /* a number ranks before NaN */
    if (!na && va != vb) return va > vb;
    return ia < ib;                   /* equal values (or both NaN): lower index */
}

/* Selection and weights from given logits (k <= n). */
int oracle_topk(const double *logits, long n, long k, long *idx, double *w)
{
    if (n < 1 || k < 1 || k > n) return -1;
    char *taken = (char *)calloc((size_t)n, 1);
    if (!taken) return -1;
    for (long r = 0; r < k; ++r) {
        long best = -1;
        for (long e = 0; e < n; ++e) {
            if (taken[e]) continue;
            if (best < 0 || ranks_before(logits[e], e, logits[best], best)) best = e;
        }
        taken[best] = 1;
        idx[r] = best;
    }
    free(taken);
    const double lmax = logits[idx[0]];
    double sum = 0.0;
    for (long r = 0; r < k; ++r) {
        w[r] = exp(logits[idx[r]] - lmax);
        sum += w[r];
    }
    for (long r = 0; r < k; ++r) w[r] /= sum;
    return 0;
}

/* logits (and sum |g x| per expert) of the bf16 router, then the selection. */
int oracle_route(const uint16_t *g, long n_experts, long d_model, const double *x, long k,
                 double *logits, double *absdot, long *idx, double *w)
{
    int rc = oracle_matvec_bf16(g, n_experts, d_model, x, 0, n_experts, logits, absdot);
    if (rc) return rc;
    return oracle_topk(logits, n_experts, k, idx, w);
}

/* out[j] = sum_i w[i] * eo[i][j] over the k rows of eo [k x d_model], in row
 * order, with sum |w[i] * eo[i][j]| per output for the tolerance. */
int oracle_combine(const double *eo, const double *w, long k, long d_model, double *out,
                   double *absdot)
{
    if (k < 0 || d_model < 0) return -1;
    for (long j = 0; j < d_model; ++j) {
        double acc = 0.0, mag = 0.0;
        for (long i = 0; i < k; ++i) {
            const double t = w[i] * eo[i * d_model + j];
            acc += t;
            mag += fabs(t);
        }
        out[j] = acc;
        if (absdot) absdot[j] = mag;
    }
    return 0;
}
