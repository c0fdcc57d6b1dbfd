// resolvent_internal.h -- launch interfaces between the C ABI (api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>

namespace rs {

constexpr int kBlock = 128;          // token block = key/query tile of the head kernel
constexpr int kMaxSlots = 128;       // heads per launch (the head table travels as a kernel parameter)
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // bound on any device-side wait: 2 s
constexpr int32_t RS_STATUS_NONFINITE_BIT = 0x1;  // same values as the public RS_STATUS_* bits
constexpr int32_t RS_STATUS_TIMEOUT_BIT = 0x2;

// Heads handled by one launch: slot -> (b*H + h, switches). Passed by value.
struct HeadTable {
    int count;
    int bh[kMaxSlots];
    float beta[kMaxSlots];
    float qk[kMaxSlots];
    float g[kMaxSlots];
};

// ---------------------------------------------------------------- gate preparation (K1)
struct GatePrepArgs {
    const float *u, *theta;
    int n;
    float *m, *theta_p;          // [BH,n] or null
    float2 *gate, *prefix, *suffix;  // [BH,n] or null
    float2 *carry;               // [BH,nb] or null
    int32_t *status;
    int write_ungated;           // 0: heads with g == 0 are only checked (nothing written)
};
cudaError_t launch_gate_prep(const GatePrepArgs &a, const HeadTable &tab, cudaStream_t s);

// ---------------------------------------------------------------- finiteness / conversion
cudaError_t launch_check_finite_bf16(const __nv_bfloat16 *x, int64_t per_head, const HeadTable &tab,
                                     int32_t *status, cudaStream_t s);
cudaError_t launch_check_finite_f32(const float *x, int64_t per_head, const HeadTable &tab,
                                    int32_t *status, cudaStream_t s);
// Rows of `cols` values (fp32 or bf16) -> rows of `dst_cols` bf16 (round to nearest even),
// zero-padded on the right. check_finite: flag non-finite source values.
cudaError_t launch_pad_to_bf16(const void *src, int src_is_f32, int64_t rows, int cols,
                               __nv_bfloat16 *dst, int dst_cols, int32_t *status,
                               int check_finite, cudaStream_t s);

// ---------------------------------------------------------------- chain scan (K3)
struct ChainArgs {
    const float *u, *theta;
    const void *b;               // fp32 or bf16 [BH,n,dv]
    int b_is_bf16;
    int n, dv;
    float *y_re, *y_im;
    int *counter;                // ticket counter (zeroed before launch)
    int *flags;                  // [slots * nchunks] (zeroed before launch)
    float2 *agg_a;               // [slots * nchunks]
    float2 *agg_y;               // [slots * nchunks * dv]
    float2 *incl_y;              // [slots * nchunks * dv]
    // normalize != 0: also run the real chain z_i = m_i z_{i-1} + 1 (z_i = sum_j R_ij) and
    // write y_i z_i^{-beta} with beta per head from the table (the qk = 0 readout)
    int normalize;
    float2 *agg_z;               // [slots * nchunks]: (prod m, z from a zero carry)
    float *incl_z;               // [slots * nchunks]: z at the end of the chunk
    // streaming: y at the end of the previous segment of each head (float2 [BH*dv], or
    // null: y_0 = b_0) and y at token n-1 written out (float2 [BH*dv], or null); with a
    // carry-in, token 0 takes its own gate, y_0 = a_0 y_{-1} + b_0
    const float2 *carry_in;
    float2 *carry_out;
    int32_t *status;
    uint64_t wait_limit_ns;
    int withhold_chunk;          // test knob: this ticket never publishes (-1: none)
};
constexpr int kChainChunk = 128;
size_t chain_scratch_bytes(int slots, int n, int dv);
cudaError_t launch_chain_scan(const ChainArgs &a, const HeadTable &tab, cudaStream_t s);
// Fixed device-side scratch for callers that cannot allocate (8 MiB).
constexpr size_t kChainNoAllocBytes = size_t(8) << 20;
// Device address of that scratch on the current device (looked up once per device).
cudaError_t chain_noalloc_scratch(void **ptr);

// ---------------------------------------------------------------- head kernel (K2)
struct HeadArgs {
    int n, d, dv;
    const float2 *gate, *prefix, *suffix, *carry;  // gate products of K1 (gated heads)
    float *O_re, *O_im;
    int32_t *status;
    int tma_out;  // O staged in shared memory and written by coalesced 16-byte stores (dv % 4 == 0); else plain stores
    int heads_per_group;  // blocks are ordered head group by head group (1 <= it <= table count)
    int *numkv;           // [slots * nqt] off-diagonal key tiles of each query tile (gated heads)
    int withhold;         // test knob: this block's K/V loads stop after its first tile (-1: none)
    int prefetch_ahead;   // this block prefetches into L2 the first tiles of block + this (0: none)
};
// The tensor maps of one head launch: q, k, v (bf16, box 64 x 128).
struct HeadMaps {
    CUtensorMap q, k, v;
};
// The number of off-diagonal key tiles of every query tile of a table of gated heads, into
// a.numkv (one warp per tile; launched right before that table's head launch).
cudaError_t launch_head_numkv(const HeadArgs &a, const HeadTable &tab, cudaStream_t s);
// dpad, dvpad in {64, 128}
cudaError_t launch_head_fwd(const HeadArgs &a, const HeadTable &tab, const HeadMaps &maps,
                            int dpad, int dvpad, cudaStream_t s);

// ---------------------------------------------------------------- materialised operator (K4)
struct OpArgs {
    int n, d;
    int chunk;                   // key tiles per row-statistics unit (operator_chunk(n))
    const float2 *gate, *prefix, *suffix, *carry;  // gate products of K1 (gated heads)
    float *W_re, *W_im;          // [BH, n, n]
    float2 *part;                // [slots, nqt, ceil(nqt / chunk), 128] partial (M, Z) per row
    float2 *ctab;                // [slots, nqt, nqt] carry products C(QB, KB)
    float4 *rowf;                // [slots, nqt * 128] (M, f, f prefix_i) per row
    float *rowq;                 // [slots, nqt * 128] |prefix_i| (1 ungated; 0 past n)
    int32_t *status;
    int tma_out;                 // W written by tensor-map stores (n % 4 == 0); else plain stores
    int withhold_stats;          // test knobs: this block of the statistics / write launch loads
    int withhold_write;          //   nothing for its second tile (-1: none)
};
// q, k (bf16, box 64 x 128) and, when tma_out is set, W_re and W_im (fp32, box 32 x 32).
struct OpMaps {
    CUtensorMap q, k, wre, wim;
};
int operator_chunk(int n);
// Multiprocessors of the current device (looked up once per device).
int device_sm_count();
// Row statistics (partials and carry products, then the merged row data: two launches),
// then W; per table of heads of one kind, in this order on one stream.
cudaError_t launch_operator_stats(const OpArgs &a, const HeadTable &tab, const OpMaps &maps, int dpad,
                                  cudaStream_t s);
cudaError_t launch_operator(const OpArgs &a, const HeadTable &tab, const OpMaps &maps, int dpad,
                            cudaStream_t s);

// ---------------------------------------------------------------- position-only heads (K5)
struct PosArgs {
    int n, H, dv;
    const float *a;              // [H, n] logit per offset d = i - j (head h of every batch reads row h)
    __nv_bfloat16 *kap;          // [slots, kstride] kappa(d) = e^{qk a(d) - M} rounded to bf16, 0 past n
    int kstride;                 // kap row stride: ceil(n / 128) * 128 + 128
    float *C;                    // [slots, n] prefix sums of the rounded kappa (scratch)
    float2 *meta;                // [slots] (M, last offset whose kappa is not 0, as int bits)
    float *O;                    // [BH, n, dv]
    int32_t *status;
    int vec_out;                 // O staged and written by 16-byte stores (dv % 4 == 0)
    int heads_per_group;         // blocks are ordered head group by head group
    int withhold;                // test knob: this block's V loads stop after its first (-1: none)
};
// v (bf16, box 64 x 128).
struct PosMaps {
    CUtensorMap v;
};
// The prep launch (kappa, prefix sums) then the main launch, per table; dvpad in {64, 128}.
cudaError_t launch_position_head(const PosArgs &a, const HeadTable &tab, const PosMaps &maps, int dvpad,
                                 cudaStream_t s);

// ---------------------------------------------------------------- debug path product
cudaError_t launch_debug_path_product(const float2 *gate, const float2 *prefix,
                                      const float2 *suffix, const float2 *carry, int n,
                                      const HeadTable &tab, float2 *G, cudaStream_t s);

}  // namespace rs
