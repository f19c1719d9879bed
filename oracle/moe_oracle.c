/*
 * moe_oracle.c -- plain, slow, fp64 CPU oracle of one Mixture-of-Experts layer
 * forward pass: router top-k/softmax, dispatch into expert-contiguous rows,
 * per-expert SwiGLU feed-forward network, gate-weighted combine.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test-suite, the smoke check and the
 * bench's CPU-baseline leg may load this library. It shares no code, header,
 * table or helper with the CUDA path and must never be called by the product.
 *
 * What it follows:
 *   - "Fine-grained Computation-Communication Overlap via Tile-level Signaling
 *     and Scheduling for MoE" (Cui et al.), section 2.1: the MoE forward is
 *     (1) routing -- top-k experts from a probability distribution, giving gate
 *     weights; (2) dispatch of each token copy to its expert; (3) expert
 *     computation; (4)-(5) return and the gate-weighted sum of the expert outputs.
 *   - "X-Stage: An Overlooked Pipeline Stage ..." (Xian et al.), section 2.2
 *     (MegaMoE Execution): each expert is Linear-1 to the intermediate width, a
 *     SwiGLU activation, Linear-2 back to the hidden width; combine aggregates
 *     the top-k results with the router weights.
 *
 * Readings where the pages give no formula (each one the plainest reading):
 *   - logits z[t,e] = sum_i x[t,i] * Wr[e,i] + b[e];
 *   - experts are selected by logit, descending, ties to the lower index; the
 *     selection is decided on fp32 logits accumulated in ascending i (each
 *     bf16*bf16 product is exact in fp32, one rounding per addition, then one
 *     for the bias), i.e. in the kernel's precision; everything else is fp64;
 *   - gates are the softmax of the k selected logits (fp64 logits);
 *   - dispatch order inside an expert is ascending (token, choice);
 *   - SwiGLU: h = silu(x W1^T) * (x W3^T), y = h W2^T, no biases.
 *
 * Parity status: every function here is pinned by the CPU tests (hand-worked
 * example, brute force, closed forms, library cross-checks, invariants).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_EINVAL 1

static double bf(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static float bf32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* ------------------------------------------------------------------------ */
/* a tiny parallel-for: items [0, n) split into contiguous blocks per thread */

typedef void (*orc_body_fn)(void *ctx, long lo, long hi);

typedef struct {
    orc_body_fn fn;
    void *ctx;
    long lo, hi;
} orc_job;

static void *orc_run(void *p)
{
    orc_job *j = (orc_job *)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

static void parallel_for(long n, int nthreads, orc_body_fn fn, void *ctx)
{
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 512) nthreads = 512;
    if (n <= 0) return;
    if ((long)nthreads > n) nthreads = (int)n;
    if (nthreads == 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t th[512];
    orc_job jobs[512];
    int started[512];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].fn = fn;
        jobs[i].ctx = ctx;
        jobs[i].lo = n * i / nthreads;
        jobs[i].hi = n * (i + 1) / nthreads;
        started[i] = pthread_create(&th[i], NULL, orc_run, &jobs[i]) == 0;
        if (!started[i]) orc_run(&jobs[i]);
    }
    for (int i = 0; i < nthreads; ++i)
        if (started[i]) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------ */
/* Step 1: routing (Cui et al. sec. 2.1 step 1; Xian et al. sec. 2.2).       */

typedef struct {
    int T, d, E, k;
    const uint16_t *x, *wr;
    const float *bias;
    int32_t *idx;
    double *gate;
    float *z32;
    double *z64;
    uint8_t *fp_sensitive;
} route_ctx;

static void route_body(void *p, long lo, long hi)
{
    route_ctx *c = (route_ctx *)p;
    const int d = c->d, E = c->E, k = c->k;
    float *zf = (float *)malloc(sizeof(float) * (size_t)E);
    double *zd = (double *)malloc(sizeof(double) * (size_t)E);
    uint8_t *taken = (uint8_t *)malloc((size_t)E);
    int32_t sel64[8];
    for (long t = lo; t < hi; ++t) {
        const uint16_t *xt = c->x + (size_t)t * d;
        for (int e = 0; e < E; ++e) {
            const uint16_t *we = c->wr + (size_t)e * d;
            float s32 = 0.0f;
            double s64 = 0.0;
            for (int i = 0; i < d; ++i) {
                float p32 = bf32(xt[i]) * bf32(we[i]); /* exact: 8-bit x 8-bit mantissas */
                s32 = s32 + p32;
                s64 += bf(xt[i]) * bf(we[i]);
            }
            if (c->bias) {
                s32 = s32 + c->bias[e];
                s64 += (double)c->bias[e];
            }
            zf[e] = s32;
            zd[e] = s64;
            if (c->z32) c->z32[(size_t)t * E + e] = s32;
            if (c->z64) c->z64[(size_t)t * E + e] = s64;
        }
        /* selection by fp32 logit, descending; ties to the lower expert index */
        memset(taken, 0, (size_t)E);
        int32_t *it = c->idx + (size_t)t * k;
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || zf[e] > zf[best]) best = e;
            }
            taken[best] = 1;
            it[j] = best;
        }
        /* same selection on the fp64 logits, only to flag fp-sensitive tokens */
        if (c->fp_sensitive) {
            memset(taken, 0, (size_t)E);
            int diff = 0;
            for (int j = 0; j < k; ++j) {
                int best = -1;
                for (int e = 0; e < E; ++e) {
                    if (taken[e]) continue;
                    if (best < 0 || zd[e] > zd[best]) best = e;
                }
                taken[best] = 1;
                sel64[j] = best;
                if (sel64[j] != it[j]) diff = 1;
            }
            c->fp_sensitive[t] = (uint8_t)diff;
        }
        /* gates: softmax over the k selected logits, fp64 */
        double zmax = zd[it[0]];
        for (int j = 1; j < k; ++j)
            if (zd[it[j]] > zmax) zmax = zd[it[j]];
        double den = 0.0;
        double num[8];
        for (int j = 0; j < k; ++j) {
            num[j] = exp(zd[it[j]] - zmax);
            den += num[j];
        }
        for (int j = 0; j < k; ++j) c->gate[(size_t)t * k + j] = num[j] / den;
    }
    free(zf);
    free(zd);
    free(taken);
}

int orc_route(int T, int d, int E, int k, const uint16_t *x, const uint16_t *wr,
              const float *bias, int32_t *topk_idx, double *topk_gate, float *z32,
              double *z64, uint8_t *fp_sensitive, int nthreads)
{
    if (T < 0 || d < 1 || E < 1 || k < 1 || k > 8 || k > E || !x || !wr || !topk_idx ||
        !topk_gate)
        return ORC_EINVAL;
    route_ctx c = {T, d, E, k, x, wr, bias, topk_idx, topk_gate, z32, z64, fp_sensitive};
    parallel_for(T, nthreads, route_body, &c);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Step 2: dispatch -- counting sort of the T*k token copies by expert,      */
/* stable in (token, choice) order (Cui et al. sec. 2.1 step 2).             */

int orc_dispatch(int T, int k, int E, const int32_t *topk_idx, int32_t *counts,
                 int32_t *offsets, int32_t *row_of_slot, int32_t *slot_of_row)
{
    if (T < 0 || k < 1 || E < 1 || !topk_idx || !counts || !offsets || !row_of_slot ||
        !slot_of_row)
        return ORC_EINVAL;
    const long R = (long)T * k;
    for (int e = 0; e < E; ++e) counts[e] = 0;
    for (long s = 0; s < R; ++s) {
        int e = topk_idx[s];
        if (e < 0 || e >= E) return ORC_EINVAL;
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t *cursor = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (long t = 0; t < T; ++t) {
        for (int j = 0; j < k; ++j) {
            long s = t * k + j;
            int e = topk_idx[s];
            int32_t r = offsets[e] + cursor[e];
            cursor[e] += 1;
            row_of_slot[s] = r;
            slot_of_row[r] = (int32_t)s;
        }
    }
    free(cursor);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Step 3: one expert's SwiGLU FFN on given input rows (Xian et al. sec 2.2). */
/* expert_kind 0 = SwiGLU FFN, 1 = identity expert (y = x).                  */

typedef struct {
    int d, F, E, kind;
    const int32_t *expert;
    const uint16_t *xin;
    const uint16_t *w1, *w3, *w2;
    double *h, *y;
} ffn_ctx;

static void ffn_one(const ffn_ctx *c, long r, double *a, double *b, double *hv)
{
    const int d = c->d, F = c->F;
    const int e = c->expert[r];
    const uint16_t *xr = c->xin + (size_t)r * d;
    double *yr = c->y + (size_t)r * d;
    if (c->kind == 1) {
        for (int o = 0; o < d; ++o) yr[o] = bf(xr[o]);
        return;
    }
    const uint16_t *W1 = c->w1 + (size_t)e * F * d;
    const uint16_t *W3 = c->w3 + (size_t)e * F * d;
    const uint16_t *W2 = c->w2 + (size_t)e * d * F;
    for (int f = 0; f < F; ++f) {
        double sa = 0.0, sb = 0.0;
        const uint16_t *g = W1 + (size_t)f * d, *u = W3 + (size_t)f * d;
        for (int i = 0; i < d; ++i) {
            double xi = bf(xr[i]);
            sa += xi * bf(g[i]);
            sb += xi * bf(u[i]);
        }
        a[f] = sa;
        b[f] = sb;
        hv[f] = sa * (1.0 / (1.0 + exp(-sa))) * sb;
        if (c->h) c->h[(size_t)r * F + f] = hv[f];
    }
    for (int o = 0; o < d; ++o) {
        const uint16_t *w = W2 + (size_t)o * F;
        double s = 0.0;
        for (int f = 0; f < F; ++f) s += hv[f] * bf(w[f]);
        yr[o] = s;
    }
}

static void ffn_body(void *p, long lo, long hi)
{
    ffn_ctx *c = (ffn_ctx *)p;
    double *a = (double *)malloc(sizeof(double) * (size_t)c->F);
    double *b = (double *)malloc(sizeof(double) * (size_t)c->F);
    double *hv = (double *)malloc(sizeof(double) * (size_t)c->F);
    for (long r = lo; r < hi; ++r) ffn_one(c, r, a, b, hv);
    free(a);
    free(b);
    free(hv);
}

int orc_ffn_rows(int d, int F, int E, long nrows, const int32_t *expert_of_row,
                 const uint16_t *xin, const uint16_t *w1, const uint16_t *w3,
                 const uint16_t *w2, double *h, double *y, int expert_kind, int nthreads)
{
    if (d < 1 || F < 1 || E < 1 || nrows < 0 || !expert_of_row || !xin || !y) return ORC_EINVAL;
    if (expert_kind == 0 && (!w1 || !w3 || !w2)) return ORC_EINVAL;
    for (long r = 0; r < nrows; ++r)
        if (expert_of_row[r] < 0 || expert_of_row[r] >= E) return ORC_EINVAL;
    ffn_ctx c = {d, F, E, expert_kind, expert_of_row, xin, w1, w3, w2, h, y};
    parallel_for(nrows, nthreads, ffn_body, &c);
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Steps 4-5: combine -- out[t] = sum_j gate[t,j] * y[row_of_slot[t*k+j]],   */
/* summed in j order (Cui et al. sec. 2.1 steps 4-5).                        */

int orc_combine(int T, int k, int d, const double *y_rows, const double *gate,
                const int32_t *row_of_slot, double *out)
{
    if (T < 0 || k < 1 || d < 1 || !y_rows || !gate || !row_of_slot || !out) return ORC_EINVAL;
    for (long t = 0; t < T; ++t) {
        double *o = out + (size_t)t * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (int j = 0; j < k; ++j) {
            const double g = gate[t * k + j];
            const double *yr = y_rows + (size_t)row_of_slot[t * k + j] * d;
            for (int c = 0; c < d; ++c) o[c] += g * yr[c];
        }
    }
    return ORC_OK;
}

/* ------------------------------------------------------------------------ */
/* Whole layer for a list of tokens, straight from the definition:           */
/* out[t] = sum_j gate[t,j] * FFN_{idx[t,j]}(x[t]).                          */

typedef struct {
    int T, d, E, k, F, kind;
    const uint16_t *x;
    const int32_t *idx;
    const double *gate;
    const uint16_t *w1, *w3, *w2;
    const int32_t *tokens;
    double *out;
} tok_ctx;

static void tok_body(void *p, long lo, long hi)
{
    tok_ctx *c = (tok_ctx *)p;
    const int d = c->d, F = c->F, k = c->k;
    double *a = (double *)malloc(sizeof(double) * (size_t)F);
    double *b = (double *)malloc(sizeof(double) * (size_t)F);
    double *hv = (double *)malloc(sizeof(double) * (size_t)F);
    double *yv = (double *)malloc(sizeof(double) * (size_t)d);
    for (long n = lo; n < hi; ++n) {
        const long t = c->tokens[n];
        double *o = c->out + (size_t)n * d;
        for (int q = 0; q < d; ++q) o[q] = 0.0;
        for (int j = 0; j < k; ++j) {
            int32_t e = c->idx[t * k + j];
            ffn_ctx fc = {d, F, c->E, c->kind, &e, c->x + (size_t)t * d, c->w1, c->w3, c->w2,
                          NULL, yv};
            ffn_one(&fc, 0, a, b, hv);
            const double g = c->gate[t * k + j];
            for (int q = 0; q < d; ++q) o[q] += g * yv[q];
        }
    }
    free(a);
    free(b);
    free(hv);
    free(yv);
}

int orc_layer_tokens(int T, int d, int E, int k, int F, const uint16_t *x,
                     const int32_t *topk_idx, const double *topk_gate, const uint16_t *w1,
                     const uint16_t *w3, const uint16_t *w2, long ntok, const int32_t *tokens,
                     double *out, int expert_kind, int nthreads)
{
    if (T < 0 || d < 1 || E < 1 || k < 1 || F < 1 || !x || !topk_idx || !topk_gate || !tokens ||
        !out || ntok < 0)
        return ORC_EINVAL;
    if (expert_kind == 0 && (!w1 || !w3 || !w2)) return ORC_EINVAL;
    for (long n = 0; n < ntok; ++n) {
        if (tokens[n] < 0 || tokens[n] >= T) return ORC_EINVAL;
        for (int j = 0; j < k; ++j) {
            int e = topk_idx[(long)tokens[n] * k + j];
            if (e < 0 || e >= E) return ORC_EINVAL;
        }
    }
    tok_ctx c = {T, d, E, k, F, expert_kind, x, topk_idx, topk_gate, w1, w3, w2, tokens, out};
    parallel_for(ntok, nthreads, tok_body, &c);
    return ORC_OK;
}
