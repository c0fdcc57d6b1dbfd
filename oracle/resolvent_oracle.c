/*
 * resolvent_oracle.c -- plain fp64 CPU oracle of the resolvent-operator causal head.
 *
 * TEST INFRASTRUCTURE: used only by the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark. It is deliberately slow and literal: explicit descending path
 * products, one row of the operator at a time, no blocking, no fusion. It shares nothing
 * with the CUDA library.
 *
 * Source of every formula: "Resolvent Operator" (teerth.dev/Aether-Lang/integrated/
 * resolvent/), section "Object" (the definition block: scaled logit, blended gate, gate,
 * path product, modulus, row normaliser, W, readout), section "Evaluation and refusals"
 * (log-domain normaliser shifted by the maximum over live entries R_ij > 0, the refusal
 * table, the zero-lane rule), section "The path-product corner is a resolvent" (the
 * chain) and the note under "Rust API" (path products accumulate from k = i down to
 * k = j+1; a_0 is never read).
 *
 * Readings where the pages leave a step open:
 *  - lerp(1, u, g) is (1-g)*1 + g*u: exact at g = 0 (gives 1) and at g = 1 (gives u).
 *  - "shifted by its maximum": the maximum of qk*s_ij over live entries (R_ij > 0).
 *  - beta*log Z is taken as 0 when beta = 0, so W = G e^{qk s} exactly at beta = 0.
 *  - a logit is refused when non-finite on any causal entry j <= i, live or not; with
 *    qk = 0 the dot product is not evaluated, so it cannot overflow (the pages accept it).
 *  - the chain starts at y_0 = b_0 (the page's y_0 = 0 is the case b_0 = 0).
 * Parity status: beta strictly inside (0,1) -- the pages give no value there; the tests pin
 * the closed forms of constant logits (W_ij = (i+1)^-beta for q = 0 and open gates, and the
 * constant-logit position head) and W(beta) * Z^beta = W(0).
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (contraction off so that x86 and
 * Arm builds round identically).
 */
#include "resolvent_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

int ro_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- gate (Object) */

int ro_blend(double u, double theta, double g, double *m, double *theta_p)
{
    /* Non-finite magnitude, phase or switch is refused ("Evaluation and refusals"). */
    if (!isfinite(u) || !isfinite(theta) || !isfinite(g)) return RO_NONFINITE;
    double l = (1.0 - g) * 1.0 + g * u;          /* lerp(1, u, g) */
    double mm = l < 0.0 ? 0.0 : (l > 1.0 ? 1.0 : l); /* clamp(., 0, 1) */
    double tp = g * theta;                       /* theta' = g theta */
    if (!isfinite(tp)) return RO_NONFINITE;      /* blended phase that overflows */
    *m = mm;
    *theta_p = tp;
    return RO_OK;
}

void ro_gate(double m, double theta_p, double *a_re, double *a_im)
{
    *a_re = m * cos(theta_p);
    *a_im = m * sin(theta_p);
}

/* complex product (xr + i xi)(yr + i yi), written out */
static void cmul(double xr, double xi, double yr, double yi, double *zr, double *zi)
{
    *zr = xr * yr - xi * yi;
    *zi = xr * yi + xi * yr;
}

/* ---------------------------------------------------------------- path product */

void ro_path_product(const double *a_re, const double *a_im, int64_t n,
                     double *G_re, double *G_im)
{
    for (int64_t i = 0; i < n; ++i) {
        double *gr = G_re + i * n, *gi = G_im + i * n;
        for (int64_t j = i + 1; j < n; ++j) { gr[j] = 0.0; gi[j] = 0.0; }
        gr[i] = 1.0; gi[i] = 0.0;                 /* G_ii = 1, the empty product */
        /* G_ij = G_i,j+1 * a_{j+1}: the product accumulates from k = i down to j+1 */
        for (int64_t j = i - 1; j >= 0; --j)
            cmul(gr[j + 1], gi[j + 1], a_re[j + 1], a_im[j + 1], &gr[j], &gi[j]);
    }
}

/* ---------------------------------------------------------------- one operator row */

typedef struct {
    double *G_re, *G_im, *R, *t;
} row_scratch;

static int scratch_alloc(row_scratch *s, int64_t n)
{
    size_t bytes = (size_t)(n > 0 ? n : 1) * sizeof(double);
    s->G_re = (double *)malloc(bytes);
    s->G_im = (double *)malloc(bytes);
    s->R = (double *)malloc(bytes);
    s->t = (double *)malloc(bytes);
    return s->G_re && s->G_im && s->R && s->t;
}

static void scratch_free(row_scratch *s)
{
    free(s->G_re); free(s->G_im); free(s->R); free(s->t);
}

/*
 * Row i of W: W_ij = G_ij exp(qk s_ij - beta log Z_i) for j <= i.
 * m, a_re, a_im: the head's gates (index 0 never read). Writes W_re/W_im[0..i].
 */
static int operator_row(const float *q, const float *k, const double *m,
                        const double *a_re, const double *a_im, int64_t d, int64_t i,
                        double beta, double qk, row_scratch *s, double *W_re, double *W_im)
{
    double *G_re = s->G_re, *G_im = s->G_im, *R = s->R, *t = s->t;

    /* path product and its modulus, k from i down to j+1 */
    G_re[i] = 1.0; G_im[i] = 0.0; R[i] = 1.0;
    for (int64_t j = i - 1; j >= 0; --j) {
        cmul(G_re[j + 1], G_im[j + 1], a_re[j + 1], a_im[j + 1], &G_re[j], &G_im[j]);
        R[j] = R[j + 1] * m[j + 1];
    }

    /* logits qk * s_ij, s_ij = <q_i, k_j> / sqrt(d); not evaluated at qk = 0 */
    const double sqrt_d = sqrt((double)d);
    for (int64_t j = 0; j <= i; ++j) {
        if (qk == 0.0) { t[j] = 0.0; continue; }
        double dot = 0.0;
        for (int64_t e = 0; e < d; ++e)
            dot += (double)q[i * d + e] * (double)k[j * d + e];
        t[j] = qk * (dot / sqrt_d);
        if (!isfinite(t[j])) return RO_NONFINITE;  /* a logit that overflows */
    }

    /* log Z_i from a sum shifted by the maximum over live entries (R_ij > 0) */
    double M = -INFINITY;
    for (int64_t j = 0; j <= i; ++j)
        if (R[j] > 0.0 && t[j] > M) M = t[j];
    double Zs = 0.0;
    for (int64_t j = 0; j <= i; ++j)
        if (R[j] > 0.0) Zs += R[j] * exp(t[j] - M);
    double logZ = M + log(Zs);

    for (int64_t j = 0; j <= i; ++j) {
        double e = exp(t[j] - (beta == 0.0 ? 0.0 : beta * logZ));
        /* a lane of G that is exactly 0 stays 0 (never 0 * inf) */
        W_re[j] = (G_re[j] == 0.0) ? 0.0 : G_re[j] * e;
        W_im[j] = (G_im[j] == 0.0) ? 0.0 : G_im[j] * e;
    }
    return RO_OK;
}

static int all_finite(const float *x, int64_t count)
{
    for (int64_t i = 0; i < count; ++i)
        if (!isfinite(x[i])) return 0;
    return 1;
}

/* gates of one head: m, a (and theta') from (u, theta, g); refusal on non-finite input */
static int head_gates(const float *u, const float *theta, double g, int64_t n,
                      double *m, double *thp, double *a_re, double *a_im)
{
    for (int64_t t = 0; t < n; ++t) {
        double mm, tp;
        int rc = ro_blend((double)u[t], (double)theta[t], g, &mm, &tp);
        if (rc != RO_OK) return rc;
        m[t] = mm;
        if (thp) thp[t] = tp;
        ro_gate(mm, tp, &a_re[t], &a_im[t]);
    }
    return RO_OK;
}

static int switches_finite(double beta, double qk, double g)
{
    return isfinite(beta) && isfinite(qk) && isfinite(g);
}

/* ---------------------------------------------------------------- operator, readout */

int ro_operator(const float *q, const float *k, const float *u, const float *theta,
                int64_t n, int64_t d, double beta, double qk, double g,
                double *W_re, double *W_im)
{
    if (n == 0) return RO_OK;                         /* empty in, empty out */
    if (n < 0 || d <= 0) return RO_SHAPE;             /* head_dim = 0 with n > 0 */
    if (!switches_finite(beta, qk, g)) return RO_NONFINITE;
    if (!all_finite(q, n * d) || !all_finite(k, n * d)) return RO_NONFINITE;

    double *m = (double *)malloc(sizeof(double) * n);
    double *a_re = (double *)malloc(sizeof(double) * n);
    double *a_im = (double *)malloc(sizeof(double) * n);
    row_scratch s;
    int ok = m && a_re && a_im && scratch_alloc(&s, n);
    int rc = ok ? head_gates(u, theta, g, n, m, NULL, a_re, a_im) : RO_SHAPE;
    for (int64_t i = 0; rc == RO_OK && i < n; ++i) {
        double *wr = W_re + i * n, *wi = W_im + i * n;
        for (int64_t j = i + 1; j < n; ++j) { wr[j] = 0.0; wi[j] = 0.0; } /* j > i */
        rc = operator_row(q, k, m, a_re, a_im, d, i, beta, qk, &s, wr, wi);
    }
    if (ok) scratch_free(&s);
    free(m); free(a_re); free(a_im);
    return rc;
}

int ro_operator_rows(const float *q, const float *k, const float *u, const float *theta,
                     int64_t n, int64_t d, double beta, double qk, double g,
                     const int64_t *rows, int64_t nrows, double *W_re, double *W_im)
{
    if (n < 0 || d <= 0 || nrows < 0) return RO_SHAPE;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= n) return RO_SHAPE;
    if (nrows == 0) return RO_OK;
    if (!switches_finite(beta, qk, g)) return RO_NONFINITE;
    if (!all_finite(q, n * d) || !all_finite(k, n * d)) return RO_NONFINITE;

    double *m = (double *)malloc(sizeof(double) * n);
    double *a_re = (double *)malloc(sizeof(double) * n);
    double *a_im = (double *)malloc(sizeof(double) * n);
    row_scratch s;
    int ok = m && a_re && a_im && scratch_alloc(&s, n);
    int rc = ok ? head_gates(u, theta, g, n, m, NULL, a_re, a_im) : RO_SHAPE;
    for (int64_t r = 0; rc == RO_OK && r < nrows; ++r) {
        const int64_t i = rows[r];
        double *wr = W_re + r * n, *wi = W_im + r * n;
        for (int64_t j = i + 1; j < n; ++j) { wr[j] = 0.0; wi[j] = 0.0; } /* j > i */
        rc = operator_row(q, k, m, a_re, a_im, d, i, beta, qk, &s, wr, wi);
    }
    if (ok) scratch_free(&s);
    free(m); free(a_re); free(a_im);
    return rc;
}

void ro_readout(const double *W_re, const double *W_im, const float *v,
                int64_t n, int64_t dv, double *O_re, double *O_im)
{
    for (int64_t i = 0; i < n; ++i) {
        double *orr = O_re + i * dv, *oi = O_im + i * dv;
        for (int64_t c = 0; c < dv; ++c) { orr[c] = 0.0; oi[c] = 0.0; }
        for (int64_t j = 0; j < n; ++j) {
            double wr = W_re[i * n + j], wi = W_im[i * n + j];
            for (int64_t c = 0; c < dv; ++c) {
                orr[c] += wr * (double)v[j * dv + c];
                oi[c] += wi * (double)v[j * dv + c];
            }
        }
    }
}

/* ---------------------------------------------------------------- chain */

void ro_chain(const double *a_re, const double *a_im, const float *b, int64_t n, int64_t dv,
              double *y_re, double *y_im, double *env)
{
    if (n <= 0) return;
    for (int64_t c = 0; c < dv; ++c) {
        y_re[c] = (double)b[c];
        y_im[c] = 0.0;
        if (env) env[c] = fabs((double)b[c]);
    }
    for (int64_t i = 1; i < n; ++i) {
        double ar = a_re[i], ai = a_im[i], am = hypot(ar, ai);
        for (int64_t c = 0; c < dv; ++c) {
            double pr = y_re[(i - 1) * dv + c], pi = y_im[(i - 1) * dv + c], zr, zi;
            cmul(ar, ai, pr, pi, &zr, &zi);            /* a_i y_{i-1} */
            y_re[i * dv + c] = zr + (double)b[i * dv + c];
            y_im[i * dv + c] = zi;
            if (env) env[i * dv + c] = am * env[(i - 1) * dv + c] + fabs((double)b[i * dv + c]);
        }
    }
}

/* ---------------------------------------------------------------- batched routines */

int ro_head_rows(const float *q, const float *k, const float *u, const float *theta,
                 const float *v, int64_t BH, int64_t n, int64_t d, int64_t dv,
                 const double *beta, const double *qk, const double *g,
                 const int64_t *rows, int64_t nrows, double *O_re, double *O_im,
                 int32_t *status, int threads)
{
    if (BH < 0 || n < 0 || nrows < 0) return RO_SHAPE;
    if (BH == 0 || n == 0) return RO_OK;
    if (d <= 0 || dv <= 0) return RO_SHAPE;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= n) return RO_SHAPE;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
    double *m = (double *)malloc(sizeof(double) * BH * n);
    double *a_re = (double *)malloc(sizeof(double) * BH * n);
    double *a_im = (double *)malloc(sizeof(double) * BH * n);
    if (!m || !a_re || !a_im) { free(m); free(a_re); free(a_im); return RO_SHAPE; }

    /* per head: refusal checks and gates */
#pragma omp parallel for schedule(dynamic)
    for (int64_t h = 0; h < BH; ++h) {
        int rc = RO_OK;
        if (!switches_finite(beta[h], qk[h], g[h])) rc = RO_NONFINITE;
        if (rc == RO_OK && (!all_finite(q + h * n * d, n * d) || !all_finite(k + h * n * d, n * d)))
            rc = RO_NONFINITE;
        if (rc == RO_OK)
            rc = head_gates(u + h * n, theta + h * n, g[h], n, m + h * n, NULL,
                            a_re + h * n, a_im + h * n);
        status[h] = rc;
    }

    /* per (head, row): one operator row, then its readout */
#pragma omp parallel
    {
        row_scratch s;
        double *wr = (double *)malloc(sizeof(double) * n);
        double *wi = (double *)malloc(sizeof(double) * n);
        int ok = scratch_alloc(&s, n) && wr && wi;
#pragma omp for schedule(dynamic)
        for (int64_t task = 0; task < BH * nrows; ++task) {
            int64_t h = task / nrows, r = task % nrows, i = rows[r];
            double *orr = O_re + (h * nrows + r) * dv, *oi = O_im + (h * nrows + r) * dv;
            for (int64_t c = 0; c < dv; ++c) { orr[c] = 0.0; oi[c] = 0.0; }
            if (!ok || status[h] != RO_OK) continue;
            const float *qh = q + h * n * d, *kh = k + h * n * d, *vh = v + h * n * dv;
            int rc = operator_row(qh, kh, m + h * n, a_re + h * n, a_im + h * n, d, i,
                                  beta[h], qk[h], &s, wr, wi);
            if (rc != RO_OK) {
#pragma omp atomic write
                status[h] = rc;
                continue;
            }
            for (int64_t j = 0; j <= i; ++j)
                for (int64_t c = 0; c < dv; ++c) {
                    orr[c] += wr[j] * (double)vh[j * dv + c];
                    oi[c] += wi[j] * (double)vh[j * dv + c];
                }
        }
        if (s.G_re || s.G_im || s.R || s.t) scratch_free(&s);
        free(wr); free(wi);
    }
    free(m); free(a_re); free(a_im);
    int rc = RO_OK;
    for (int64_t h = 0; h < BH; ++h)
        if (status[h] != RO_OK) rc = status[h];
    return rc;
}

int ro_gate_prep(const float *u, const float *theta, const double *g, int64_t BH, int64_t n,
                 int64_t block, double *m, double *theta_p, double *a_re, double *a_im,
                 double *pre_re, double *pre_im, double *suf_re, double *suf_im,
                 double *car_re, double *car_im, int32_t *status)
{
    if (BH < 0 || n < 0 || block <= 0) return RO_SHAPE;
    const int64_t nb = (n + block - 1) / block;
    int rc_all = RO_OK;
#pragma omp parallel for schedule(dynamic)
    for (int64_t h = 0; h < BH; ++h) {
        double *hm = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
        double *ht = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
        double *ar = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
        double *ai = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
        int rc = (hm && ht && ar && ai) ? RO_OK : RO_SHAPE;
        if (rc == RO_OK && !isfinite(g[h])) rc = RO_NONFINITE;
        if (rc == RO_OK) rc = head_gates(u + h * n, theta + h * n, g[h], n, hm, ht, ar, ai);
        status[h] = rc;
        if (rc == RO_OK) {
            for (int64_t t = 0; t < n; ++t) {
                if (m) m[h * n + t] = hm[t];
                if (theta_p) theta_p[h * n + t] = ht[t];
                if (a_re) a_re[h * n + t] = ar[t];
                if (a_im) a_im[h * n + t] = ai[t];
            }
            for (int64_t b = 0; b < nb; ++b) {
                int64_t s = b * block, e = s + block - 1 < n - 1 ? s + block - 1 : n - 1;
                int64_t lo = s > 1 ? s : 1;               /* a_0 is never read */
                for (int64_t i = s; i <= e; ++i) {
                    /* prefix: prod_{k=lo..i} a_k, accumulated from k = i down */
                    double pr = 1.0, pi = 0.0;
                    for (int64_t kk = i; kk >= lo; --kk) cmul(pr, pi, ar[kk], ai[kk], &pr, &pi);
                    /* suffix: prod_{k=i+1..e} a_k, accumulated from k = e down */
                    double sr = 1.0, si = 0.0;
                    for (int64_t kk = e; kk >= i + 1; --kk) cmul(sr, si, ar[kk], ai[kk], &sr, &si);
                    if (pre_re) pre_re[h * n + i] = pr;
                    if (pre_im) pre_im[h * n + i] = pi;
                    if (suf_re) suf_re[h * n + i] = sr;
                    if (suf_im) suf_im[h * n + i] = si;
                }
                double cr = 1.0, ci = 0.0;
                for (int64_t kk = e; kk >= lo; --kk) cmul(cr, ci, ar[kk], ai[kk], &cr, &ci);
                if (car_re) car_re[h * nb + b] = cr;
                if (car_im) car_im[h * nb + b] = ci;
            }
        }
        free(hm); free(ht); free(ar); free(ai);
    }
    for (int64_t h = 0; h < BH; ++h)
        if (status[h] != RO_OK) rc_all = status[h];
    return rc_all;
}

int ro_chain_heads(const float *u, const float *theta, const double *g, const float *b,
                   int64_t BH, int64_t n, int64_t dv, double *y_re, double *y_im,
                   double *env, int32_t *status, int threads)
{
    if (BH < 0 || n < 0 || dv <= 0) return RO_SHAPE;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
#pragma omp parallel for schedule(dynamic)
    for (int64_t h = 0; h < BH; ++h) {
        double *m = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
        double *ar = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
        double *ai = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
        int rc = (m && ar && ai) ? RO_OK : RO_SHAPE;
        if (rc == RO_OK && !isfinite(g[h])) rc = RO_NONFINITE;
        if (rc == RO_OK) rc = head_gates(u + h * n, theta + h * n, g[h], n, m, NULL, ar, ai);
        status[h] = rc;
        if (rc == RO_OK)
            ro_chain(ar, ai, b + h * n * dv, n, dv, y_re + h * n * dv, y_im + h * n * dv,
                     env ? env + h * n * dv : NULL);
        free(m); free(ar); free(ai);
    }
    int rc = RO_OK;
    for (int64_t h = 0; h < BH; ++h)
        if (status[h] != RO_OK) rc = status[h];
    return rc;
}

/* Position-only head: the definition row by row (see the header). */
/* Row i of a position-only head from the logits t[d] = qk a(d) of every offset: a softmax
 * row of t[i - j], j <= i, with Z_i taken from the sum shifted by the row maximum (every
 * entry is live), O_i = sum_j e^{t[i-j]} v_j / Z_i^beta. */
static void position_row(const double *t, const float *v, int64_t i, int64_t dv, double beta,
                         double *Orow)
{
    double M = -INFINITY;
    for (int64_t j = 0; j <= i; ++j)
        if (t[i - j] > M) M = t[i - j];
    double Zs = 0.0;
    for (int64_t j = 0; j <= i; ++j) Zs += exp(t[i - j] - M);
    const double logZ = M + log(Zs);
    for (int64_t c = 0; c < dv; ++c) Orow[c] = 0.0;
    for (int64_t j = 0; j <= i; ++j) {
        const double w = exp(t[i - j] - (beta == 0.0 ? 0.0 : beta * logZ));
        for (int64_t c = 0; c < dv; ++c) Orow[c] += w * (double)v[j * dv + c];
    }
}

/* The logits of every offset, refusing a non-finite a(d) (even at qk = 0) or qk a(d);
 * NULL after a refusal (*rc set) or when out of memory. */
static double *position_logits(const float *a, int64_t n, double qk, int *rc)
{
    *rc = RO_OK;
    if (!all_finite(a, n)) {
        *rc = RO_NONFINITE;
        return NULL;
    }
    double *t = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!t) {
        *rc = RO_SHAPE;
        return NULL;
    }
    for (int64_t d = 0; d < n; ++d) {
        t[d] = qk * (double)a[d];  /* the logit of every pair at offset d */
        if (!isfinite(t[d])) {
            free(t);
            *rc = RO_NONFINITE;
            return NULL;
        }
    }
    return t;
}

int ro_position_head(const float *a, const float *v, int64_t n, int64_t dv, double beta,
                     double qk, double *O)
{
    if (n == 0) return RO_OK;
    if (n < 0 || dv <= 0) return RO_SHAPE;
    if (!isfinite(beta) || !isfinite(qk)) return RO_NONFINITE;
    int rc;
    double *t = position_logits(a, n, qk, &rc);
    if (!t) return rc;
    for (int64_t i = 0; i < n; ++i) position_row(t, v, i, dv, beta, O + i * dv);
    free(t);
    return RO_OK;
}

int ro_position_rows(const float *a, const float *v, int64_t n, int64_t dv, double beta,
                     double qk, const int64_t *rows, int64_t nrows, double *O)
{
    if (n < 0 || dv <= 0 || nrows < 0) return RO_SHAPE;
    for (int64_t k = 0; k < nrows; ++k)
        if (rows[k] < 0 || rows[k] >= n) return RO_SHAPE;
    if (nrows == 0) return RO_OK;
    if (!isfinite(beta) || !isfinite(qk)) return RO_NONFINITE;
    int rc;
    double *t = position_logits(a, n, qk, &rc);
    if (!t) return rc;
    for (int64_t k = 0; k < nrows; ++k) position_row(t, v, rows[k], dv, beta, O + k * dv);
    free(t);
    return RO_OK;
}

int ro_position_heads(const float *a, const float *v, int64_t BH, int64_t H, int64_t n,
                      int64_t dv, const double *beta, const double *qk, double *O,
                      int32_t *status, int threads)
{
    if (BH < 0 || H <= 0 || n < 0 || dv <= 0) return RO_SHAPE;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif
#pragma omp parallel for schedule(dynamic)
    for (int64_t h = 0; h < BH; ++h)
        status[h] = ro_position_head(a + (h % H) * n, v + h * n * dv, n, dv, beta[h], qk[h],
                                     O + h * n * dv);
    int rc = RO_OK;
    for (int64_t h = 0; h < BH; ++h)
        if (status[h] != RO_OK) rc = status[h];
    return rc;
}
