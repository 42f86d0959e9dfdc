/*
 * oracle.c -- plain, slow, single-threaded fp64 oracle for the GQA attention
 * hot path of a greedy Qwen3-style decoder.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header, table or constant with the
 * CUDA library; it reads its inputs as fp64 values (exact images of the bf16
 * inputs) and computes everything in fp64 with libm.
 *
 * What it computes, and where the pages say so:
 *   - per-head RMSNorm of q and k, then rotary embedding ("RMSNorm, rotary
 *     embedding and the attention epilogue are small, repeated, and safe to
 *     fuse" -- dryft-flash-infer agent guide, section "Where the wins are");
 *   - append of the transformed k and the raw v into a preallocated cache, one
 *     slot per (sequence, kv head, position) (same guide, "Where the wins are",
 *     KV-cache-layout bullet: a preallocated, correctly strided cache);
 *   - causal grouped-query softmax attention over the whole prompt (prefill,
 *     same section, prefill bullet) and over the cache for one new token
 *     (decode step, same section, per-step-overhead bullet);
 *   - cache reset per generate call (same guide, "What is measured").
 * The pages name the Qwen3 model but print no formula; the formulas below are
 * the textbook definitions of that family and the readings are:
 *   RMSNorm    y_i = w_i * x_i / sqrt(mean_j x_j^2 + eps)          (weight multiplies directly)
 *   RoPE       rotate-half pairs (i, i + D/2), angle a_i = pos * theta^(-2i/D),
 *              x'_i = x_i cos a_i - x_{i+D/2} sin a_i,
 *              x'_{i+D/2} = x_{i+D/2} cos a_i + x_i sin a_i
 *   attention  out = sum_j softmax_j(q . k_j / sqrt(D)) v_j over j <= own position,
 *              q head h reads kv head floor(h / G), G = Hq / Hkv
 *   positions  each sequence starts at position 0 (packed, unpadded batches)
 *   decode     the new token is appended first and attends to itself.
 * The score row is materialised in full; there is no tiling, no online
 * softmax and no split of the key range.
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

/* Status codes of the oracle (its own, unrelated to the library's). */
#define ORACLE_OK 0
#define ORACLE_BAD_ARG 1
#define ORACLE_OVERFLOW 2
#define ORACLE_NO_MEMORY 3

/* RMSNorm of one head vector x[D] with weight w[D]. */
void oracle_rmsnorm(int D, const double *x, const double *w, double eps, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < D; ++i)
        ss += x[i] * x[i];
    double r = sqrt(ss / (double)D + eps);
    for (int i = 0; i < D; ++i)
        y[i] = w[i] * x[i] / r;
}

/* Rotate-half rotary embedding of one head vector x[D] at position pos. */
void oracle_rope(int D, double pos, double theta, const double *x, double *y)
{
    int half = D / 2;
    for (int i = 0; i < half; ++i) {
        double a = pos * pow(theta, -2.0 * (double)i / (double)D);
        double c = cos(a), s = sin(a);
        double x1 = x[i], x2 = x[i + half];
        y[i] = x1 * c - x2 * s;
        y[i + half] = x2 * c + x1 * s;
    }
}

/*
 * Softmax attention of one query q[D] over n keys: K row j at K + j*stride,
 * V row j at V + j*stride.  Writes out[D]; if p is not NULL it also receives
 * the n softmax weights.
 */
int oracle_attend(int D, int n, const double *q, const double *K, const double *V,
                  long stride, double *out, double *p)
{
    if (n <= 0 || D <= 0)
        return ORACLE_BAD_ARG;
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    if (!s)
        return ORACLE_NO_MEMORY;
    double scale = 1.0 / sqrt((double)D);
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += q[d] * K[(long)j * stride + d];
        s[j] = dot * scale;
        if (s[j] > m)
            m = s[j];
    }
    double l = 0.0;
    for (int j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    for (int d = 0; d < D; ++d)
        out[d] = 0.0;
    for (int j = 0; j < n; ++j) {
        double pj = s[j] / l;
        if (p)
            p[j] = pj;
        for (int d = 0; d < D; ++d)
            out[d] += pj * V[(long)j * stride + d];
    }
    free(s);
    return ORACLE_OK;
}

/*
 * Geometry of one attention layer as the oracle sees it.  Its cache is its
 * own fp64 array Kc/Vc[B][Hkv][cap][D]; lens[B] are the cached lengths.
 */
typedef struct {
    int B, Hq, Hkv, D, cap;
    double theta, eps;
} oracle_geom;

static long cache_row(const oracle_geom *g, int b, int kvh, int pos)
{
    return (((long)b * g->Hkv + kvh) * g->cap + pos) * g->D;
}

/*
 * Transform and append a packed prompt batch: sequence b holds tokens
 * [cu_b, cu_b + plen[b]) of q[T][Hq][D], k[T][Hkv][D], v[T][Hkv][D], where cu_b
 * is the sum of the earlier lengths.  Writes qp[T][Hq][D] (normed, rotated q),
 * fills cache slots 0..plen[b]-1 of every kv head with the normed, rotated k
 * and the raw v, and sets lens[b] = plen[b].  Requires lens[b] == 0 (an
 * empty layer) and plen[b] <= cap.
 */
int oracle_prefill_transform(const oracle_geom *g, const int *plen,
                             const double *q, const double *k, const double *v,
                             const double *wq, const double *wk,
                             double *qp, double *Kc, double *Vc, int *lens)
{
    int D = g->D;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)D);
    if (!tmp)
        return ORACLE_NO_MEMORY;
    long t = 0;
    for (int b = 0; b < g->B; ++b) {
        if (plen[b] < 0 || plen[b] > g->cap || lens[b] != 0) {
            free(tmp);
            return plen[b] > g->cap ? ORACLE_OVERFLOW : ORACLE_BAD_ARG;
        }
        for (int i = 0; i < plen[b]; ++i, ++t) {
            for (int h = 0; h < g->Hq; ++h) {
                const double *x = q + (t * g->Hq + h) * D;
                oracle_rmsnorm(D, x, wq, g->eps, tmp);
                oracle_rope(D, (double)i, g->theta, tmp, qp + (t * g->Hq + h) * D);
            }
            for (int h = 0; h < g->Hkv; ++h) {
                const double *x = k + (t * g->Hkv + h) * D;
                oracle_rmsnorm(D, x, wk, g->eps, tmp);
                oracle_rope(D, (double)i, g->theta, tmp, Kc + cache_row(g, b, h, i));
                memcpy(Vc + cache_row(g, b, h, i), v + (t * g->Hkv + h) * D,
                       sizeof(double) * (size_t)D);
            }
        }
        lens[b] = plen[b];
    }
    free(tmp);
    return ORACLE_OK;
}

/*
 * Causal attention output of one prompt row: query qp_row[D] of sequence b,
 * head h, at position i, over cache slots 0..i of kv head floor(h / G).
 */
int oracle_prefill_row(const oracle_geom *g, int b, int h, int i,
                       const double *qp_row, const double *Kc, const double *Vc,
                       double *out)
{
    if (b < 0 || b >= g->B || h < 0 || h >= g->Hq || i < 0 || i >= g->cap)
        return ORACLE_BAD_ARG;
    int G = g->Hq / g->Hkv;
    int kvh = h / G;
    return oracle_attend(g->D, i + 1, qp_row, Kc + cache_row(g, b, kvh, 0),
                         Vc + cache_row(g, b, kvh, 0), g->D, out, NULL);
}

/* Whole prefill of one layer: transform + append, then every output row. */
int oracle_prefill(const oracle_geom *g, const int *plen,
                   const double *q, const double *k, const double *v,
                   const double *wq, const double *wk,
                   double *qp, double *Kc, double *Vc, int *lens, double *out)
{
    int rc = oracle_prefill_transform(g, plen, q, k, v, wq, wk, qp, Kc, Vc, lens);
    if (rc != ORACLE_OK)
        return rc;
    long t = 0;
    for (int b = 0; b < g->B; ++b)
        for (int i = 0; i < plen[b]; ++i, ++t)
            for (int h = 0; h < g->Hq; ++h) {
                rc = oracle_prefill_row(g, b, h, i, qp + (t * g->Hq + h) * g->D, Kc, Vc,
                                        out + (t * g->Hq + h) * g->D);
                if (rc != ORACLE_OK)
                    return rc;
            }
    return ORACLE_OK;
}

/*
 * Transform and append the new token of every sequence: the token of
 * sequence b sits at position pos = lens[b]; its q and k are normed and
 * rotated at pos, k' and the raw v go to slot pos, and lens[b] becomes
 * pos + 1.  q[B][Hq][D], k/v[B][Hkv][D]; writes qp[B][Hq][D].  A full cache
 * (lens[b] == cap) is an error: nothing is evicted or wrapped.
 */
int oracle_decode_transform(const oracle_geom *g, const double *q, const double *k,
                            const double *v, const double *wq, const double *wk,
                            double *Kc, double *Vc, int *lens, double *qp)
{
    int D = g->D;
    for (int b = 0; b < g->B; ++b)
        if (lens[b] < 0 || lens[b] >= g->cap)
            return lens[b] >= g->cap ? ORACLE_OVERFLOW : ORACLE_BAD_ARG;
    double *tmp = (double *)malloc(sizeof(double) * (size_t)D);
    if (!tmp)
        return ORACLE_NO_MEMORY;
    for (int b = 0; b < g->B; ++b) {
        int pos = lens[b];
        for (int h = 0; h < g->Hkv; ++h) {
            oracle_rmsnorm(D, k + ((long)b * g->Hkv + h) * D, wk, g->eps, tmp);
            oracle_rope(D, (double)pos, g->theta, tmp, Kc + cache_row(g, b, h, pos));
            memcpy(Vc + cache_row(g, b, h, pos), v + ((long)b * g->Hkv + h) * D,
                   sizeof(double) * (size_t)D);
        }
        for (int h = 0; h < g->Hq; ++h) {
            oracle_rmsnorm(D, q + ((long)b * g->Hq + h) * D, wq, g->eps, tmp);
            oracle_rope(D, (double)pos, g->theta, tmp, qp + ((long)b * g->Hq + h) * D);
        }
        lens[b] = pos + 1;
    }
    free(tmp);
    return ORACLE_OK;
}

/*
 * One decode step for every sequence: transform and append as above, then
 * every q head attends over slots 0..pos of its kv head (the new token
 * attends to itself).  Writes qp[B][Hq][D] and out[B][Hq][D].
 */
int oracle_decode(const oracle_geom *g, const double *q, const double *k, const double *v,
                  const double *wq, const double *wk,
                  double *Kc, double *Vc, int *lens, double *qp, double *out)
{
    int D = g->D, G = g->Hq / g->Hkv;
    int rc = oracle_decode_transform(g, q, k, v, wq, wk, Kc, Vc, lens, qp);
    if (rc != ORACLE_OK)
        return rc;
    for (int b = 0; b < g->B; ++b) {
        int n = lens[b];
        for (int h = 0; h < g->Hq; ++h) {
            rc = oracle_attend(D, n, qp + ((long)b * g->Hq + h) * D,
                               Kc + cache_row(g, b, h / G, 0), Vc + cache_row(g, b, h / G, 0), D,
                               out + ((long)b * g->Hq + h) * D, NULL);
            if (rc != ORACLE_OK)
                return rc;
        }
    }
    return ORACLE_OK;
}

/* Reset for a new generate call: lengths to zero; cache contents are kept. */
void oracle_reset(const oracle_geom *g, int *lens)
{
    for (int b = 0; b < g->B; ++b)
        lens[b] = 0;
}
