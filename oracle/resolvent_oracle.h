/*
 * resolvent_oracle.h -- plain fp64 CPU oracle of the resolvent-operator causal head.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark call this library. It shares no code, header, helper or constant with
 * the CUDA library under gated_causal_attention_gb300/csrc, and the product path never
 * loads it.
 *
 * Every routine follows the definition block of "Resolvent Operator"
 * (teerth.dev/Aether-Lang/integrated/resolvent/, section "Object") and the evaluation rule
 * of its section "Evaluation and refusals". Arithmetic is IEEE fp64 throughout. Inputs
 * that the GPU reads as bf16 or fp32 are passed here as fp32 arrays holding the very same
 * stored values (bf16 -> fp32 -> fp64 is exact), so both sides see identical numbers.
 *
 * Layout: row-major and contiguous. A "head" is one (batch, head) slice; batched routines
 * take BH heads laid out one after another: q,k [BH,n,d], v,b [BH,n,dv], u,theta [BH,n].
 * Complex outputs are split planes (re, im) of the same shape.
 *
 * Return codes: RO_OK, RO_NONFINITE (the pages' NonFinite refusal), RO_SHAPE (shape error,
 * which the pages' Rust module signals by panicking).
 *
 * Parity status: every routine is pinned by the CPU test suite against closed forms,
 * library routines and the pages' printed values. For beta strictly inside (0,1), where the
 * pages give no value, the pins are the closed forms of constant logits (W_ij = (i+1)^-beta
 * for q = 0 and open gates; the constant-logit position head) and W(beta) * Z^beta == W(0).
 */
#ifndef RESOLVENT_ORACLE_H
#define RESOLVENT_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { RO_OK = 0, RO_NONFINITE = 1, RO_SHAPE = 2 };

/* Blended gate ("Object", blended-gate row; Rust API `blend`):
 * m = clamp(lerp(1, u, g), 0, 1) with lerp(1,u,g) = (1-g)*1 + g*u, theta' = g*theta. */
int ro_blend(double u, double theta, double g, double *m, double *theta_p);

/* The gate ("Object", gate row; Rust API `gate`): a = m * e^{i theta'}. */
void ro_gate(double m, double theta_p, double *a_re, double *a_im);

/* Path product ("Object", path-product row; Rust API `path_product`):
 * G[i,j] = prod_{k=j+1..i} a_k for j <= i (accumulated from k = i down to k = j+1),
 * G[i,i] = 1, G[i,j] = 0 for j > i. a_0 is never read. G is [n,n] row-major. */
void ro_path_product(const double *a_re, const double *a_im, int64_t n,
                     double *G_re, double *G_im);

/* Operator W [n,n] ("Object", W row, evaluated per "Evaluation and refusals"). */
int ro_operator(const float *q, const float *k, const float *u, const float *theta,
                int64_t n, int64_t d, double beta, double qk, double g,
                double *W_re, double *W_im);

/* Rows rows[0 .. nrows) of the same operator (each 0 <= rows[k] < n), W_re/W_im [nrows, n]:
 * the same per-row arithmetic as ro_operator, for sampled checks at large n. */
int ro_operator_rows(const float *q, const float *k, const float *u, const float *theta,
                     int64_t n, int64_t d, double beta, double qk, double g,
                     const int64_t *rows, int64_t nrows, double *W_re, double *W_im);

/* Readout ("Object", readout row; Rust API `readout`): O_i = sum_j W_ij V_j. */
void ro_readout(const double *W_re, const double *W_im, const float *v,
                int64_t n, int64_t dv, double *O_re, double *O_im);

/* Chain ("The path-product corner is a resolvent"; Rust API `chain_label`):
 * y_0 = b_0, y_i = a_i y_{i-1} + b_i. The page states the chain for b_0 = 0, where y_0 = 0;
 * starting from b_0 makes it the path-product readout for any b. b is [n,dv] real,
 * y is [n,dv] complex. Also returns the forward-error envelope
 * env_i = |a_i| env_{i-1} + |b_i| (env may be NULL). */
void ro_chain(const double *a_re, const double *a_im, const float *b, int64_t n, int64_t dv,
              double *y_re, double *y_im, double *env);

/* Batched head readout at selected rows, without materialising W:
 * O[h, r, :] = sum_{j <= rows[r]} W_{rows[r], j} V_j for head h, with per-head switches
 * beta[h], qk[h], g[h]. Output [BH, nrows, dv]. status[h] receives the head's code.
 * Parallel over (head, row) with OpenMP when built with it; threads <= 0 uses the default. */
int ro_head_rows(const float *q, const float *k, const float *u, const float *theta,
                 const float *v, int64_t BH, int64_t n, int64_t d, int64_t dv,
                 const double *beta, const double *qk, const double *g,
                 const int64_t *rows, int64_t nrows, double *O_re, double *O_im,
                 int32_t *status, int threads);

/* Batched gate preparation on blocks of `block` tokens. For block b = [s, e]:
 *   prefix[i] = prod_{k=max(s,1)..i} a_k   (inclusive, from the block's first token)
 *   suffix[j] = prod_{k=j+1..e} a_k       (exclusive; 1 at j = e)
 *   carry[b]  = prod_{k=max(s,1)..e} a_k  (the whole block)
 * all accumulated from the highest index down, like the path product, and a_0 never read.
 * These are entries of the path product: prefix[i] = G[i, s-1], suffix[j] = G[e, j],
 * carry[b] = G[e, s-1] (with s-1 read as 0 for the first block).
 * Any output pointer may be NULL. Shapes: m, theta_p [BH,n]; gate/prefix/suffix complex
 * [BH,n]; carry complex [BH, ceil(n/block)]. status[h] receives the head's code. */
int ro_gate_prep(const float *u, const float *theta, const double *g, int64_t BH, int64_t n,
                 int64_t block, double *m, double *theta_p, double *a_re, double *a_im,
                 double *pre_re, double *pre_im, double *suf_re, double *suf_im,
                 double *car_re, double *car_im, int32_t *status);

/* Batched chain over heads, gates from (u, theta, g): y [BH,n,dv] complex, env [BH,n,dv]. */
int ro_chain_heads(const float *u, const float *theta, const double *g, const float *b,
                   int64_t BH, int64_t n, int64_t dv, double *y_re, double *y_im,
                   double *env, int32_t *status, int threads);

/* Threads the OpenMP runtime would use (1 when built without OpenMP). */
int ro_max_threads(void);

/* Position-only head: "A position-only causal softmax head is a causal convolution divided
 * by a prefix normalizer" (proofs.blah.dev, theorem pos-head-is-causal-convolution), its
 * left-hand side, with the switches of "Resolvent Operator" at g = 0 (no gates, so every
 * entry is live): the logit of query i and key j is t_ij = qk * a(i - j),
 * W_ij = e^{t_ij} / Z_i^beta with Z_i = sum_{j<=i} e^{t_ij}, evaluated in the log domain of
 * "Evaluation and refusals" (log Z_i = M_i + log sum_j e^{t_ij - M_i}, M_i = max_j t_ij), and
 * O_i = sum_{j<=i} W_ij v_j. a [n] (one logit per offset d = i - j), v [n,dv], O [n,dv], all
 * real. Refusals: a non-finite a(d) for d < n (even at qk = 0, as q and k are refused there),
 * a non-finite switch, a non-finite qk * a(d). */
int ro_position_head(const float *a, const float *v, int64_t n, int64_t dv, double beta,
                     double qk, double *O);

/* Rows rows[0 .. nrows) of the same head (each 0 <= rows[k] < n), O [nrows, dv]: the same
 * per-row arithmetic as ro_position_head, for sampled checks of long sequences. */
int ro_position_rows(const float *a, const float *v, int64_t n, int64_t dv, double beta,
                     double qk, const int64_t *rows, int64_t nrows, double *O);

/* The same for BH heads: head h reads its offset logits at a + (h % H) * n (a [H,n], one
 * table per head index, shared across the batch), v [BH,n,dv], switches beta[h], qk[h];
 * O [BH,n,dv]. status[h] receives the head's code. Parallel over heads with OpenMP. */
int ro_position_heads(const float *a, const float *v, int64_t BH, int64_t H, int64_t n,
                      int64_t dv, const double *beta, const double *qk, double *O,
                      int32_t *status, int threads);

#ifdef __cplusplus
}
#endif
#endif
