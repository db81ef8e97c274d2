/*
 * Oracle for the PowerInfer hot path: activation predictor -> neuron-aware
 * sparse FFN, one layer and one decode step at a time.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * CPU statement of what the GPU library computes.  Only the test-suite, the
 * smoke check and the benchmark's CPU-baseline leg may load it.  It shares no
 * code, header, table or helper with the CUDA library, and the library never
 * calls it.
 *
 * Sources (PowerInfer: Fast LLM Serving with a Consumer-grade GPU):
 *   - chatpaper.ai abstract: "adaptive predictors and neuron-aware sparse
 *     operators"; hot/cold neurons from a power-law activation distribution.
 *   - blog.csdn.net (QbitAI/IPADS), section "充分利用模型和硬件特点": about 10%
 *     of OPT FFN neurons suffice; a small per-layer routing predictor decides,
 *     before the FFN runs, which neurons the input activates, and only those
 *     neurons are computed.
 *   - same page, section "CPU/GPU混合推理设计": worked example, predicted set
 *     {3,4,5}; the two executors compute disjoint parts and the partial
 *     results are merged.
 *   - de.news.hada.io summary, "Quantisierung und Kompatibilität": Q4_0 INT4.
 * The pages print no formulas.  The readings this file implements (canonical
 * fp32 dot order, z > 0 threshold, Q4_0 block layout, weightless RMSNorm
 * between layers) are listed in the design notes beside the code.
 *
 * Precision: every FFN quantity is fp64.  The predictor is evaluated in fp32
 * in one fixed operation order (CDOT below) so that the active set is a
 * deterministic function of the input bytes; it also reports the fp64 value
 * of every predictor logit so that near-threshold margins can be inspected.
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared (no fast-math).  fmaf() is
 * the C library's correctly rounded fused multiply-add.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { OR_F16 = 0, OR_BF16 = 1, OR_Q4_0 = 2 };
enum { OR_RELU = 0, OR_REGLU = 1, OR_SQRELU = 2 };
enum { OR_OK = 0, OR_EARG = -1 };

/* ------------------------------------------------------------------ */
/* Number formats (IEEE 754 binary16, bfloat16, Q4_0 blocks)           */
/* ------------------------------------------------------------------ */

static double f16_value(uint16_t h)
{
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 1024), e - 25); /* 1.m * 2^(e-15) */
    return s ? -v : v;
}

static double bf16_value(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16; /* bf16 is the top half of binary32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double or_to_double(uint16_t bits, int dt)
{
    return dt == OR_BF16 ? bf16_value(bits) : f16_value(bits);
}

/* Round a double to the nearest binary16 (ties to even). */
static uint16_t round_f16(double v)
{
    if (isnan(v)) return 0x7e00;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a >= 65520.0) return sign | 0x7c00; /* half-way to 2^16 and above */
    if (a < ldexp(1.0, -14)) {              /* subnormal quantum 2^-24 */
        double q = nearbyint(ldexp(a, 24));
        return sign | (uint16_t)q; /* q == 1024 is the smallest normal */
    }
    int e;
    frexp(a, &e);
    int E = e - 1; /* a in [2^E, 2^(E+1)) */
    double q = nearbyint(ldexp(a, 10 - E)); /* in [1024, 2048] */
    if (q == 2048.0) { q = 1024.0; E += 1; }
    if (E > 15) return sign | 0x7c00;
    return sign | (uint16_t)((E + 15) << 10) | (uint16_t)((int)q - 1024);
}

/* Round a double to the nearest bfloat16 (ties to even). */
static uint16_t round_bf16(double v)
{
    if (isnan(v)) return 0x7fc0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a >= ldexp(2.0 - ldexp(1.0, -8), 127)) return sign | 0x7f80;
    if (a < ldexp(1.0, -126)) { /* subnormal quantum 2^-133 */
        double q = nearbyint(ldexp(a, 133));
        return sign | (uint16_t)q;
    }
    int e;
    frexp(a, &e);
    int E = e - 1;
    double q = nearbyint(ldexp(a, 7 - E)); /* in [128, 256] */
    if (q == 256.0) { q = 128.0; E += 1; }
    if (E > 127) return sign | 0x7f80;
    return sign | (uint16_t)((E + 127) << 7) | (uint16_t)((int)q - 128);
}

uint16_t or_round(double v, int dt)
{
    return dt == OR_BF16 ? round_bf16(v) : round_f16(v);
}

/* Q4_0 block of 32 weights: 2-byte little-endian fp16 scale s, then 16 bytes;
 * element j < 16 is the low nibble of byte j, element j >= 16 the high nibble
 * of byte j-16; the weight is (q - 8) * s. */
#define Q4_BLOCK_BYTES 18
static double q4_elem(const uint8_t *blk, int j)
{
    double s = f16_value((uint16_t)(blk[0] | (blk[1] << 8)));
    int q = j < 16 ? (blk[2 + j] & 15) : (blk[2 + j - 16] >> 4);
    return (double)(q - 8) * s;
}

void or_q4_dequant(const uint8_t *blocks, long nblocks, double *out)
{
    for (long b = 0; b < nblocks; ++b)
        for (int j = 0; j < 32; ++j)
            out[b * 32 + j] = q4_elem(blocks + b * Q4_BLOCK_BYTES, j);
}

/* Weight (row i, column k) of a matrix stored row-major with rows of length
 * `cols`, either 16-bit floats or Q4_0 blocks along the row. */
static double wval(const void *w, int dt, long cols, long i, long k)
{
    if (dt == OR_Q4_0) {
        const uint8_t *row = (const uint8_t *)w + i * (cols / 32) * Q4_BLOCK_BYTES;
        return q4_elem(row + (k / 32) * Q4_BLOCK_BYTES, (int)(k % 32));
    }
    return or_to_double(((const uint16_t *)w)[i * cols + k], dt);
}

/* ------------------------------------------------------------------ */
/* A tiny static thread pool: rows i = t, t+T, t+2T, ... go to thread t. */
/* Each output is produced by one thread in a fixed order, so results do */
/* not depend on the thread count.                                      */
/* ------------------------------------------------------------------ */

typedef void (*row_fn)(void *ctx, long i);
typedef struct { row_fn fn; void *ctx; long n; int t, nt; } par_job;

static void *par_worker(void *p)
{
    par_job *j = (par_job *)p;
    for (long i = j->t; i < j->n; i += j->nt) j->fn(j->ctx, i);
    return NULL;
}

static void par_for(long n, int nthreads, row_fn fn, void *ctx)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (nthreads == 1 || n < 2) {
        for (long i = 0; i < n; ++i) fn(ctx, i);
        return;
    }
    pthread_t th[256];
    par_job jobs[256];
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = (par_job){fn, ctx, n, t, nthreads};
        if (pthread_create(&th[t], NULL, par_worker, &jobs[t]) != 0) break;
        started++;
    }
    /* any thread that could not start: run its share here */
    for (int t = started; t < nthreads; ++t) par_worker(&jobs[t]);
    for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
}

/* ------------------------------------------------------------------ */
/* Predictor                                                           */
/* ------------------------------------------------------------------ */

/* CDOT: the canonical fp32 dot product of a 16-bit row w[0..K) with an fp32
 * vector v.  32 lanes; lane l starts at +0 and walks chunks c = l, l+32, ...
 * of 8 consecutive elements, accumulating acc = fma(w, v, acc) element by
 * element (correctly rounded).  The lanes are then combined by a butterfly:
 * for m = 16, 8, 4, 2, 1 every lane adds the old value of lane l^m (fp32,
 * round to nearest).  The result is lane 0's value. */
float or_cdot(const uint16_t *w, int dt, const float *v, int K)
{
    float lane[32], next[32];
    int nchunks = (K + 7) / 8;
    for (int l = 0; l < 32; ++l) {
        float acc = 0.0f;
        for (int c = l; c < nchunks; c += 32)
            for (int e = 0; e < 8 && 8 * c + e < K; ++e)
                acc = fmaf((float)or_to_double(w[8 * c + e], dt), v[8 * c + e], acc);
        lane[l] = acc;
    }
    for (int m = 16; m >= 1; m >>= 1) {
        for (int l = 0; l < 32; ++l) next[l] = lane[l] + lane[l ^ m];
        memcpy(lane, next, sizeof lane);
    }
    return lane[0];
}

typedef struct {
    int d, n, r, dt, B;
    const uint16_t *W1, *b1, *W2, *b2, *xhat;
    float *xf, *h;   /* B*d, B*r */
    double *h64;     /* B*r */
    float *z;        /* B*n */
    double *z64;     /* B*n */
    uint8_t *mask;   /* B*n */
} pred_ctx;

/* Hidden layer: h_j = max(CDOT(W1[j], x) + b1_j, 0) in fp32 (not rounded to
 * 16 bits), plus the fp64 value of the same quantity. */
static void pred_hidden_row(void *p, long j)
{
    pred_ctx *c = (pred_ctx *)p;
    float b = c->b1 ? (float)or_to_double(c->b1[j], c->dt) : 0.0f;
    double b64 = c->b1 ? or_to_double(c->b1[j], c->dt) : 0.0;
    for (int t = 0; t < c->B; ++t) {
        float s = or_cdot(c->W1 + j * (long)c->d, c->dt, c->xf + (long)t * c->d, c->d) + b;
        c->h[(long)t * c->r + j] = s > 0.0f ? s : 0.0f;
        double s64 = b64;
        for (int k = 0; k < c->d; ++k)
            s64 += or_to_double(c->W1[j * (long)c->d + k], c->dt) * (double)c->xf[(long)t * c->d + k];
        c->h64[(long)t * c->r + j] = s64 > 0.0 ? s64 : 0.0;
    }
}

/* Output layer: z_i = CDOT(W2[i], h) + b2_i; neuron i is predicted active
 * iff sigmoid(z_i) > 0.5, i.e. iff z_i > 0 (so +0, -0 and NaN are inactive). */
static void pred_out_row(void *p, long i)
{
    pred_ctx *c = (pred_ctx *)p;
    float b = c->b2 ? (float)or_to_double(c->b2[i], c->dt) : 0.0f;
    double b64 = c->b2 ? or_to_double(c->b2[i], c->dt) : 0.0;
    for (int t = 0; t < c->B; ++t) {
        float z = or_cdot(c->W2 + i * (long)c->r, c->dt, c->h + (long)t * c->r, c->r) + b;
        double z64 = b64;
        for (int k = 0; k < c->r; ++k)
            z64 += or_to_double(c->W2[i * (long)c->r + k], c->dt) * c->h64[(long)t * c->r + k];
        c->z[(long)t * c->n + i] = z;
        c->z64[(long)t * c->n + i] = z64;
        c->mask[(long)t * c->n + i] = z > 0.0f;
    }
}

/* Per-token predicted masks for B tokens.  h_out, z_out, z64_out may be NULL. */
int or_predict(int d, int n, int r, int dt, const uint16_t *W1, const uint16_t *b1,
               const uint16_t *W2, const uint16_t *b2, const uint16_t *xhat, int B,
               float *h_out, float *z_out, double *z64_out, uint8_t *mask, int nthreads)
{
    if (d < 1 || n < 1 || r < 1 || B < 1 || !W1 || !W2 || !xhat || !mask) return OR_EARG;
    if (dt != OR_F16 && dt != OR_BF16) return OR_EARG;
    pred_ctx c = {d, n, r, dt, B, W1, b1, W2, b2, xhat, NULL, NULL, NULL, NULL, NULL, mask};
    c.xf = malloc(sizeof(float) * (size_t)B * d);
    c.h = malloc(sizeof(float) * (size_t)B * r);
    c.h64 = malloc(sizeof(double) * (size_t)B * r);
    c.z = z_out ? z_out : malloc(sizeof(float) * (size_t)B * n);
    c.z64 = z64_out ? z64_out : malloc(sizeof(double) * (size_t)B * n);
    if (!c.xf || !c.h || !c.h64 || !c.z || !c.z64) return OR_EARG;
    for (long k = 0; k < (long)B * d; ++k) c.xf[k] = (float)or_to_double(xhat[k], dt);
    par_for(r, nthreads, pred_hidden_row, &c);
    par_for(n, nthreads, pred_out_row, &c);
    if (h_out) memcpy(h_out, c.h, sizeof(float) * (size_t)B * r);
    free(c.xf);
    free(c.h);
    free(c.h64);
    if (!z_out) free(c.z);
    if (!z64_out) free(c.z64);
    return OR_OK;
}

/* Hot neurons: the one-device reading of the hot/cold split ("CPU/GPU混合推理设计",
 * CSDN page): the listed neurons (the first ones of the calibrated order) are
 * active for every token, whatever the predictor says; the others keep their
 * predicted bit. */
int or_force_active(uint8_t *mask, int B, int n, const int32_t *ids, int nids)
{
    if (!mask || B < 1 || n < 1 || nids < 0 || (nids > 0 && !ids)) return OR_EARG;
    for (int k = 0; k < nids; ++k)
        if (ids[k] < 0 || ids[k] >= n) return OR_EARG;
    for (int t = 0; t < B; ++t)
        for (int k = 0; k < nids; ++k) mask[(long)t * n + ids[k]] = 1;
    return OR_OK;
}

/* Union over B tokens of the per-token masks, as an ascending index list. */
int or_union(const uint8_t *mask, int B, int n, int32_t *idx, int32_t *count)
{
    int m = 0;
    for (int i = 0; i < n; ++i) {
        int any = 0;
        for (int t = 0; t < B; ++t) any |= mask[(long)t * n + i] != 0;
        if (any) idx[m++] = i;
    }
    *count = m;
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* FFN (fp64)                                                          */
/* ------------------------------------------------------------------ */

typedef struct {
    int d, n, act, wdt, adt, B;
    const void *Wup, *Wgate;
    const uint16_t *b;
    const double *x; /* B*d */
    double *a;       /* B*n */
} act_ctx;

/* ReLU:         a_i = max(W_up[i].x + b_i, 0)
 * ReGLU:        a_i = max(W_gate[i].x + b_i, 0) * (W_up[i].x)      (bias on the gate)
 * Squared ReLU: a_i = max(W_up[i].x + b_i, 0)^2  (the third family the engine
 *               serves: de.news.hada.io summary, "Einschränkungen und FAQ") */
static void act_row(void *p, long i)
{
    act_ctx *c = (act_ctx *)p;
    double bi = c->b ? or_to_double(c->b[i], c->adt) : 0.0;
    for (int t = 0; t < c->B; ++t) {
        const double *x = c->x + (long)t * c->d;
        double up = 0.0;
        for (long k = 0; k < c->d; ++k) up += wval(c->Wup, c->wdt, c->d, i, k) * x[k];
        double a;
        if (c->act == OR_REGLU) {
            double g = bi;
            for (long k = 0; k < c->d; ++k) g += wval(c->Wgate, c->wdt, c->d, i, k) * x[k];
            a = (g > 0.0 ? g : 0.0) * up;
        } else {
            up += bi;
            a = up > 0.0 ? up : 0.0;
            if (c->act == OR_SQRELU) a = a * a;
        }
        c->a[(long)t * c->n + i] = a;
    }
}

/* Dense activations a[B][n] of every neuron.  Wup/Wgate: [n][d] 16-bit rows,
 * or Q4_0 blocks along each row when wdt == OR_Q4_0. */
int or_ffn_act(int d, int n, int act, int wdt, int adt, const void *Wup, const void *Wgate,
               const uint16_t *b, const uint16_t *xhat, int B, double *a, int nthreads)
{
    if (d < 1 || n < 1 || B < 1 || !Wup || !xhat || !a) return OR_EARG;
    if (act == OR_REGLU && !Wgate) return OR_EARG;
    if (wdt == OR_Q4_0 && d % 32) return OR_EARG;
    act_ctx c = {d, n, act, wdt, adt, B, Wup, Wgate, b, NULL, a};
    double *x = malloc(sizeof(double) * (size_t)B * d);
    if (!x) return OR_EARG;
    for (long k = 0; k < (long)B * d; ++k) x[k] = or_to_double(xhat[k], adt);
    c.x = x;
    par_for(n, nthreads, act_row, &c);
    free(x);
    return OR_OK;
}

typedef struct {
    int d, n, wdt, adt, B, count;
    const void *Wd;
    const uint16_t *bd;
    const double *a;
    const int32_t *idx;
    double *y;
} down_ctx;

/* y_t[j] = sum over the list (in list order) of a_t[i] * W_down[j][i], + b_down[j]. */
static void down_col(void *p, long j)
{
    down_ctx *c = (down_ctx *)p;
    double bj = c->bd ? or_to_double(c->bd[j], c->adt) : 0.0;
    for (int t = 0; t < c->B; ++t) {
        double s = 0.0;
        for (int k = 0; k < c->count; ++k) {
            long i = c->idx[k];
            /* dense W_down is [d][n] (row j, column i); Q4_0 W_down is stored
             * transposed, blocks along d in each neuron row i */
            double w = c->wdt == OR_Q4_0 ? wval(c->Wd, c->wdt, c->d, i, j)
                                         : wval(c->Wd, c->wdt, c->n, j, i);
            s += c->a[(long)t * c->n + i] * w;
        }
        c->y[(long)t * c->d + j] = s + bj;
    }
}

int or_ffn_down(int d, int n, int wdt, int adt, const void *Wdown, const uint16_t *bdown,
                const double *a, int B, const int32_t *idx, int count, double *y, int nthreads)
{
    if (d < 1 || n < 1 || B < 1 || count < 0 || count > n || !Wdown || !a || !y) return OR_EARG;
    if (count > 0 && !idx) return OR_EARG;
    for (int k = 0; k < count; ++k)
        if (idx[k] < 0 || idx[k] >= n) return OR_EARG;
    down_ctx c = {d, n, wdt, adt, B, count, Wdown, bdown, a, idx, y};
    par_for(d, nthreads, down_col, &c);
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Between layers: weightless RMSNorm of the fp32 residual stream,      */
/* x_hat = round(x / sqrt(mean(x^2) + eps)) computed in fp64.           */
/* ------------------------------------------------------------------ */
int or_rmsnorm(const float *x, int B, int d, int dt, double eps, uint16_t *xhat)
{
    if (B < 1 || d < 1 || !x || !xhat) return OR_EARG;
    for (int t = 0; t < B; ++t) {
        double ss = 0.0;
        for (int k = 0; k < d; ++k) ss += (double)x[(long)t * d + k] * (double)x[(long)t * d + k];
        double inv = 1.0 / sqrt(ss / d + eps);
        for (int k = 0; k < d; ++k)
            xhat[(long)t * d + k] = or_round((double)x[(long)t * d + k] * inv, dt);
    }
    return OR_OK;
}

/* ------------------------------------------------------------------ */
/* Offline neuron permutation: physical order = descending activation   */
/* count, ties broken by the lower original id.  perm[p] = original id. */
/* ------------------------------------------------------------------ */
static const int32_t *g_counts;
static int cmp_hot(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    if (g_counts[a] != g_counts[b]) return g_counts[a] > g_counts[b] ? -1 : 1;
    return a < b ? -1 : (a > b);
}

int or_perm_from_counts(const int32_t *counts, int n, int32_t *perm)
{
    if (n < 1 || !counts || !perm) return OR_EARG;
    for (int i = 0; i < n; ++i) perm[i] = i;
    g_counts = counts; /* single-threaded use only */
    qsort(perm, (size_t)n, sizeof(int32_t), cmp_hot);
    return OR_OK;
}
