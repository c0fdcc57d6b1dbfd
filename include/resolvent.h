/*
 * resolvent.h -- C ABI of the GB300 (sm_103a) resolvent-operator causal head.
 *
 * The operation is the one causal attention head of "Resolvent Operator"
 * (teerth.dev/Aether-Lang/integrated/resolvent/), section "Object": for 0 <= j <= i < n
 *
 *   s_ij = <q_i, k_j> / sqrt(d)                         scaled logit
 *   m_k  = clamp(lerp(1, u_k, g), 0, 1),  theta'_k = g theta_k     blended gate
 *   a_k  = m_k e^{i theta'_k}                            the gate
 *   G_ij = prod_{k=j+1..i} a_k  (G_ii = 1),  R_ij = |G_ij|           path product, modulus
 *   Z_i  = sum_{j<=i} R_ij e^{qk s_ij}                   row normaliser
 *   W_ij = G_ij e^{qk s_ij} / Z_i^beta  (j <= i),  0 above           weight
 *   O_i  = sum_{j<=i} W_ij V_j                           readout (complex; V real)
 *
 * evaluated in the log domain of section "Evaluation and refusals" (Z from a sum shifted by
 * the maximum over live entries R_ij > 0), with the refusals of that section. The chain of
 * section "The path-product corner is a resolvent" (y_i = a_i y_{i-1} + b_i) is the
 * readout at the corner (beta, qk, g) = (0, 0, 1).
 *
 * Conventions shared by every entry point
 *  - Device pointers unless stated otherwise; the caller owns every buffer. The library
 *    never allocates or frees memory and never synchronises, except in
 *    resolvent_status_sync. Scratch lives in the caller's workspace.
 *  - Layout: row-major and contiguous. A head is one (batch, head) slice bh = b*H + h:
 *    q, k [B,H,n,d]; v, b [B,H,n,dv]; u, theta [B,H,n]; O_re, O_im, y_re, y_im [B,H,n,dv].
 *    Complex per-token arrays (gate, prefix, suffix, block carry) hold interleaved
 *    (re, im) fp32 pairs.
 *  - Alignment: every pointer 16-byte aligned; head_forward also needs d % 8 == 0.
 *  - Switches (rs_switches) are HOST arrays of `count` values, count 1 (all heads) or H
 *    (value h serves head h of every batch). Non-finite switches are refused at once.
 *  - Errors found from arguments are returned synchronously. Errors that depend on the
 *    data (the pages' NonFinite refusal; a bounded wait that ran out) are OR-ed into the
 *    caller's device status word `status_dev` (one int32, zero before the first call) and
 *    read back by resolvent_status_sync. Outputs are unspecified when a refusal is raised.
 *  - n == 0 or B*H == 0 is an empty call: RS_OK, nothing launched ("Evaluation and
 *    refusals", empty sequence).
 *  - `stream` is a cudaStream_t (0 = the legacy default stream); every launch goes there.
 */
#ifndef RESOLVENT_H
#define RESOLVENT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RS_OK = 0,
    RS_ERR_NONFINITE = 1,   /* the pages' NonFinite: a non-finite input, switch, g*theta or logit */
    RS_ERR_SHAPE = 2,       /* negative sizes, d = 0 or dv = 0 with n > 0, bad switch count */
    RS_ERR_UNSUPPORTED = 3, /* a size this build does not handle (d or dv > 128, d % 8 != 0) */
    RS_ERR_ALIGN = 4,       /* a pointer that is not 16-byte aligned */
    RS_ERR_WORKSPACE = 5,   /* workspace missing or smaller than the *_workspace_bytes query */
    RS_ERR_CUDA = 6,        /* a CUDA runtime call failed (launch, tensor map, memset) */
    RS_ERR_TIMEOUT = 7      /* a bounded device-side wait ran out (reported via status_dev) */
} rs_status;

typedef enum { RS_F32 = 0, RS_BF16 = 1 } rs_dtype;

/* Per-head switches (beta, qk, g) -- the Rust API's `Switches`. Host arrays. */
typedef struct {
    const float *beta;
    const float *qk;
    const float *g;
    int count;
} rs_switches;

/* Device status-word bits (OR-ed by kernels). */
#define RS_STATUS_NONFINITE 0x1
#define RS_STATUS_TIMEOUT 0x2

/* Token block of the gate products (the key/query tile of the head kernel). */
#define RS_BLOCK 128

/*
 * Gate preparation ("Object", blended-gate and gate rows; Rust API `blend`, `gate`) and
 * the block products that factor the path product ("Object", path-product row):
 * for each head and each block [s, e] of RS_BLOCK tokens (the last one ragged)
 *   m[t] = clamp((1-g) + g u_t, 0, 1),  theta_p[t] = g theta_t,  gate[t] = a_t
 *   prefix[i] = prod_{k=max(s,1)..i} a_k       (inclusive, from the block's first token)
 *   suffix[j] = prod_{k=j+1..e} a_k           (exclusive; 1 at j = e)
 *   block_carry[b] = prod_{k=max(s,1)..e} a_k (the whole block)
 * so that for j < s(QB) <= i the path product is
 *   G_ij = prefix[i] * (prod of block_carry over the blocks strictly between) * suffix[j].
 * Gates are only multiplied (never divided or taken through a log), so a closed gate gives
 * exact zeros. a_0 is never read. Shapes: m, theta_p [B,H,n] fp32; gate, prefix, suffix
 * [B,H,n] complex; block_carry [B,H,ceil(n/RS_BLOCK)] complex. Any output may be NULL.
 * Non-finite u, theta, or an overflowing g*theta sets RS_STATUS_NONFINITE.
 */
rs_status resolvent_gate_prep(const float *u, const float *theta, rs_switches sw,
                              int B, int H, int n,
                              float *m, float *theta_p, float *gate, float *prefix,
                              float *suffix, float *block_carry,
                              int32_t *status_dev, void *stream);

/* Workspace bytes resolvent_head_forward needs for these sizes (0 when n == 0). */
size_t resolvent_head_workspace_bytes(int B, int H, int n, int d, int dv, rs_dtype dtype);

/*
 * The head: O = W V with W from section "Object" (Rust API `operator` then `readout`,
 * fused, batched over B*H heads, per-head switches). q, k [B,H,n,d] and v [B,H,n,dv] are
 * bf16 (dtype RS_BF16) or fp32 (RS_F32: rounded to bf16 into the workspace first);
 * u, theta fp32 [B,H,n]; O_re, O_im fp32 [B,H,n,dv]. The contractions run on the tensor
 * cores in bf16 with fp32 accumulation. Heads with qk = 0 are evaluated in O(n): then
 * W_ij = G_ij / Z_i^beta with Z_i = sum_{j<=i} R_ij = m_i Z_{i-1} + 1, so O_i = y_i Z_i^-beta
 * with y the chain over V (at beta = 0, W = G exactly and O = y).
 * Supported: 1 <= d <= 128 with d % 8 == 0, 1 <= dv <= 128.
 * Refusals (RS_STATUS_NONFINITE): non-finite q, k, u, theta, g*theta, or a non-finite
 * logit qk*s_ij on an evaluated entry (every diagonal entry is evaluated, so any
 * non-finite q or k row is caught). Outputs past the range of fp32 read +-inf, not NaN.
 */
rs_status resolvent_head_forward(const void *q, const void *k, const float *u,
                                 const float *theta, const void *v, rs_switches sw,
                                 int B, int H, int n, int d, int dv, rs_dtype dtype,
                                 float *O_re, float *O_im,
                                 void *workspace, size_t workspace_bytes,
                                 int32_t *status_dev, void *stream);

/* Workspace bytes resolvent_operator needs for these sizes (0 when n == 0). */
size_t resolvent_operator_workspace_bytes(int B, int H, int n, int d, rs_dtype dtype);

/*
 * The operator itself, section "Object" (Rust API `operator`): W_ij = G_ij e^{qk s_ij} / Z_i^beta
 * for every head, with the log-domain normaliser and the refusals of section "Evaluation and
 * refusals". q, k [B,H,n,d] bf16 (RS_BF16) or fp32 (RS_F32: rounded to bf16 first); u, theta
 * fp32 [B,H,n]; W_re, W_im fp32 [B,H,n,n] row-major (entry (i, j) of head (b, h) at
 * ((b*H + h)*n + i)*n + j), every entry written: 0 above the diagonal and wherever G is
 * exactly 0. The logits come from the tensor cores (bf16 inputs, fp32 accumulation); the
 * rest is fp32. Caller-owned device memory, 16-byte aligned; workspace of at least
 * resolvent_operator_workspace_bytes. Supported: 1 <= d <= 128 with d % 8 == 0.
 * Errors as for resolvent_head_forward; refusals through the status word.
 */
rs_status resolvent_operator(const void *q, const void *k, const float *u, const float *theta,
                             rs_switches sw, int B, int H, int n, int d, rs_dtype dtype,
                             float *W_re, float *W_im, void *workspace, size_t workspace_bytes,
                             int32_t *status_dev, void *stream);

/* Workspace bytes resolvent_position_head needs for these sizes (0 when n == 0). */
size_t resolvent_position_workspace_bytes(int B, int H, int n, int dv, rs_dtype dtype);

/*
 * Position-only heads: "A position-only causal softmax head is a causal convolution divided
 * by a prefix normalizer" (proofs.blah.dev, theorem pos-head-is-causal-convolution), with the
 * switches of "Resolvent Operator" at g = 0. The logit of query i and key j is qk * a_h(i - j):
 *     O_i = sum_{j<=i} e^{qk a(i-j)} v_j / Z_i^beta,  Z_i = sum_{d<=i} e^{qk a(d)},
 * evaluated as the theorem's right-hand side: a causal convolution of v with the kernel
 * kappa(d) = e^{qk a(d) - M} (M the head's largest logit; kappa rounded to bf16 for the tensor
 * cores) over the prefix sum of the same rounded kernel, times e^{(1-beta) M}. No logit is
 * formed per entry. a fp32 [H,n] (row h serves head h of every batch); v [B,H,n,dv] bf16
 * (RS_BF16) or fp32 (RS_F32: rounded to bf16 first); O fp32 [B,H,n,dv] (real: no gates).
 * beta and qk per head from the switches; every g must be 0 (else RS_ERR_UNSUPPORTED).
 * Supported: 1 <= dv <= 128. Caller-owned device memory, 16-byte aligned.
 * Refusals (RS_STATUS_NONFINITE): a non-finite a(d) (even at qk = 0) or qk * a(d), and a row
 * whose kernel values all underflow in fp32 (logits spread over more than ~87 nats in one
 * head). Errors as for resolvent_head_forward.
 */
rs_status resolvent_position_head(const float *a, const void *v, rs_switches sw, int B, int H,
                                  int n, int dv, rs_dtype dtype, float *O, void *workspace,
                                  size_t workspace_bytes, int32_t *status_dev, void *stream);

/* Workspace bytes resolvent_chain_scan needs for these sizes (0 when n == 0). */
size_t resolvent_chain_workspace_bytes(int B, int H, int n, int dv);

/*
 * The chain of section "The path-product corner is a resolvent" (Rust API `chain_label`):
 * y_0 = b_0, y_i = a_i y_{i-1} + b_i with a_i the gate of (u_i, theta_i, g) -- i.e. the
 * readout G b of the path product. The page states it for b_0 = 0, where y_0 = 0.
 * b fp32 [B,H,n,dv]; y_re, y_im fp32 [B,H,n,dv]; 1 <= dv <= 128. Only g is read from the
 * switches (the chain is the (0,0,1) corner whatever beta and qk say).
 * Single pass: chunks of tokens publish their carries to later chunks; every wait on a
 * carry is bounded, and one that runs out sets RS_STATUS_TIMEOUT.
 */
rs_status resolvent_chain_scan(const float *u, const float *theta, rs_switches sw,
                               const float *b, int B, int H, int n, int dv,
                               float *y_re, float *y_im,
                               void *workspace, size_t workspace_bytes,
                               int32_t *status_dev, void *stream);

/*
 * The same chain over one segment of a longer sequence (the resolvent applied across calls,
 * as the page's block summaries carry a prefix from block to block): carry_in holds, per head,
 * y at the end of the previous segment, and then token 0 takes its own gate,
 * y_0 = a_0 y_{-1} + b_0; carry_out receives y at token n-1. Both are interleaved complex
 * fp32 [B,H,dv] (re, im pairs), device memory owned by the caller, 16-byte aligned; either
 * may be NULL (no carry-in: y_0 = b_0 as in resolvent_chain_scan; no carry-out: nothing
 * written). carry_out may not alias carry_in. Chaining segments S1, S2, ... with carry_out of
 * one as carry_in of the next gives the chain of the concatenated sequence up to rounding.
 * Other arguments, layout and errors are those of resolvent_chain_scan. This entry has no
 * counterpart on the pages (they state the chain for one whole sequence).
 */
rs_status resolvent_chain_scan_carry(const float *u, const float *theta, rs_switches sw,
                                     const float *b, int B, int H, int n, int dv,
                                     const float *carry_in, float *carry_out,
                                     float *y_re, float *y_im,
                                     void *workspace, size_t workspace_bytes,
                                     int32_t *status_dev, void *stream);

/*
 * resolvent_chain_scan without a workspace argument: the same chain, with its scratch in a
 * fixed 8 MiB array of device memory inside this library. (The pages have no counterpart;
 * this entry exists for callers, not for the method.)
 *
 * Who needs it: callers that cannot call cudaMalloc or hand out extra device memory, e.g.
 * code that runs inside a framework whose own pool owns all device memory and forbids side
 * allocations, plugin hosts that pass only input and output buffers, or latency-critical
 * loops where an allocation (and the synchronisation it can imply) is not acceptable.
 *
 * Limit: the sizes must need at most 8 MiB of chain scratch, i.e.
 * resolvent_chain_workspace_bytes(B, H, n, dv) <= 8 MiB (about 1M tokens of B*H*n per 128
 * heads at dv = 64); larger calls return RS_ERR_UNSUPPORTED and launch nothing.
 * The array is part of this library's device code: it is reserved in a device's memory when
 * that code is loaded there and held until the process exits. Under CUDA's lazy module
 * loading (the default) that happens at the first call on the device that needs it, so in a
 * process whose memory pool will take all device memory, make the first call of this entry
 * point before the pool does, or the load can fail (RS_ERR_CUDA). The first
 * call on a device also looks up the array's device address (one cudaGetSymbolAddress with
 * that device current); make it before any stream capture. The address is kept per device
 * and context, and looked up again in a new context (after cudaDeviceReset).
 * Nothing is allocated or freed, by this library or any library it calls. The counters that
 * must start at zero are cleared on the stream at the start of every call; the rest keeps
 * the last call's contents. All calls share the one array, so calls that overlap on the GPU
 * (other streams, other threads) race: serialise them.
 * Arguments, layout, errors and results are those of resolvent_chain_scan.
 */
rs_status resolvent_chain_scan_noalloc(const float *u, const float *theta, rs_switches sw,
                                       const float *b, int B, int H, int n, int dv,
                                       float *y_re, float *y_im,
                                       int32_t *status_dev, void *stream);

/* Synchronises `stream`, reads the status word, clears it to 0 and returns RS_OK,
 * RS_ERR_TIMEOUT or RS_ERR_NONFINITE (RS_ERR_CUDA if the runtime reports an error). A timeout
 * takes precedence: after one the outputs, and any refusal raised from them, are unspecified. */
rs_status resolvent_status_sync(int32_t *status_dev, void *stream);

/* Static text for a status code. */
const char *resolvent_status_string(rs_status s);

/* Number of kernel launches the last call on this host thread enqueued (for reporting). */
int resolvent_last_launch_count(void);

/*
 * Debug export (tests only): the path product G [B,H,n,n] complex (interleaved) as the
 * head kernel factors it -- prefix x block carries x suffix across blocks, explicit
 * products inside a block -- from the gates of (u, theta, g). n <= 4096.
 */
rs_status resolvent_debug_path_product(const float *u, const float *theta, rs_switches sw,
                                       int B, int H, int n, float *G,
                                       void *workspace, size_t workspace_bytes,
                                       int32_t *status_dev, void *stream);

/*
 * Test knobs (tests only; they change how later calls on any thread behave):
 *  - the bound on device-side waits in the chain scan, in nanoseconds (0 restores 2 s);
 *  - a chain chunk ticket that never publishes its carry (-1: none), so that the bounded
 *    wait of the chunks after it runs out and RS_STATUS_TIMEOUT is raised without a hang;
 *  - a block of the position-head kernel whose V loads stop after its first (-1: none): its
 *    tensor-core issuer's wait for the next V tile runs out (2 s), RS_STATUS_TIMEOUT is
 *    raised, every block winds down (each waits for the copies and products it started) and
 *    the call returns;
 *  - the same for a block of the fused head kernel, whose K and V loads stop after its first
 *    key tile (-1: none);
 *  - the same for a block of the operator's statistics launch (launch 0) or write launch
 *    (launch 1), which loads nothing for its second tile (block -1: none).
 */
void resolvent_test_set_wait_limit_ns(uint64_t ns);
void resolvent_test_set_chain_withhold(int ticket);
void resolvent_test_set_position_withhold(int block);
void resolvent_test_set_head_withhold(int block);
void resolvent_test_set_operator_withhold(int launch, int block);

/*
 * Kernel timing (benchmarking): while enabled, each call records pairs of CUDA events on its
 * stream around its main launches, one pair per class below: each table of gated heads
 * (the key-tile count and the fused head kernel), each table of g = 0 heads, the O(n)
 * readout of qk = 0 heads, the chain scan, the operator's write of W, the position heads
 * (prep and main launch), gate preparation. resolvent_profile_collect waits for the
 * recorded pairs, writes their durations in milliseconds (at most `max`), returns how many,
 * and starts a new series (-1 on a CUDA error); resolvent_profile_collect_kinds also writes
 * each pair's class. Enabling (re)starts the series. Up to 4096 pairs are kept.
 */
#define RS_PROF_HEAD_GATED 0
#define RS_PROF_HEAD_REAL 1
#define RS_PROF_READOUT 2
#define RS_PROF_CHAIN 3
#define RS_PROF_OPERATOR 4
#define RS_PROF_POSITION 5
#define RS_PROF_GATE_PREP 6
rs_status resolvent_profile_enable(int on);
int resolvent_profile_collect(float *ms, int max);
int resolvent_profile_collect_kinds(float *ms, int *kind, int max);

#ifdef __cplusplus
}
#endif
#endif
