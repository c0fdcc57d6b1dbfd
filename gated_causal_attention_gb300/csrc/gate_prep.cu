// gate_prep.cu -- blended gates and their block products (K1), input checks, fp32 -> bf16
// rounding, and the debug export of the path product.
//
// "Resolvent Operator", section "Object": m_k = clamp(lerp(1, u_k, g), 0, 1),
// theta'_k = g theta_k, a_k = m_k e^{i theta'_k}; section "Evaluation and refusals":
// non-finite magnitudes, phases and blended phases are refused.
//
// One warp owns one block of 128 tokens; each lane holds 4 consecutive tokens. The block's
// inclusive prefix products, exclusive suffix products and total come from lane-local
// products plus a 5-step warp-shuffle scan. Gates are only multiplied.
#include "gate_products.cuh"

namespace rs {

namespace {

constexpr int kTokPerLane = kBlock / 32;  // 4

__global__ void __launch_bounds__(128)
gate_prep_kernel(GatePrepArgs a, const __grid_constant__ HeadTable tab)
{
    const int n = a.n;
    const int nb = (n + kBlock - 1) / kBlock;
    const int warp = blockIdx.x * 4 + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    const int slot = warp / nb, blk = warp % nb;
    if (slot >= tab.count) return;
    const int64_t bh = tab.bh[slot];
    const float g = tab.g[slot];
    const int64_t base = bh * (int64_t)n;
    const int t0 = blk * kBlock + lane * kTokPerLane;
    const bool write = a.write_ungated || g != 0.f;

    float uu[kTokPerLane], tt[kTokPerLane];
    if ((n & 3) == 0 && t0 + kTokPerLane <= n) {
        const float4 u4 = *reinterpret_cast<const float4 *>(a.u + base + t0);
        const float4 t4 = *reinterpret_cast<const float4 *>(a.theta + base + t0);
        uu[0] = u4.x; uu[1] = u4.y; uu[2] = u4.z; uu[3] = u4.w;
        tt[0] = t4.x; tt[1] = t4.y; tt[2] = t4.z; tt[3] = t4.w;
    } else {
#pragma unroll
        for (int k = 0; k < kTokPerLane; ++k) {
            const bool in = t0 + k < n;
            uu[k] = in ? a.u[base + t0 + k] : 1.f;
            tt[k] = in ? a.theta[base + t0 + k] : 0.f;
        }
    }

    bool bad = false;
    float mm[kTokPerLane], tp[kTokPerLane];
    cplx gt[kTokPerLane];  // the gate a_t
    cplx pg[kTokPerLane];  // the factor the products use: a_t, or 1 at t = 0 and past n
#pragma unroll
    for (int k = 0; k < kTokPerLane; ++k) {
        const int t = t0 + k;
        const float l = fmaf(g, uu[k], 1.f - g);  // lerp(1, u, g) = (1-g) + g u
        mm[k] = fminf(fmaxf(l, 0.f), 1.f);
        tp[k] = g * tt[k];
        bad |= t < n && (!isfinite(uu[k]) || !isfinite(tt[k]) || !isfinite(tp[k]));
        float sn, cs;
        sincosf(tp[k], &sn, &cs);
        gt[k] = {mm[k] * cs, mm[k] * sn};
        pg[k] = (t == 0 || t >= n) ? cplx{1.f, 0.f} : gt[k];
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(a.status, RS_STATUS_NONFINITE_BIT);
    if (!write) return;

    // lane-local inclusive prefix and exclusive suffix products
    cplx lp[kTokPerLane], ls[kTokPerLane];
    lp[0] = pg[0];
#pragma unroll
    for (int k = 1; k < kTokPerLane; ++k) lp[k] = cmul(lp[k - 1], pg[k]);
    ls[kTokPerLane - 1] = {1.f, 0.f};
#pragma unroll
    for (int k = kTokPerLane - 2; k >= 0; --k) ls[k] = cmul(ls[k + 1], pg[k + 1]);
    const cplx total = lp[kTokPerLane - 1];

    // warp scans of the lane totals: inclusive from the left, inclusive from the right
    cplx incl = total, sincl = total;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const cplx x = shfl_up(incl, d);
        if (lane >= d) incl = cmul(x, incl);
        const cplx y = shfl_down(sincl, d);
        if (lane + d < 32) sincl = cmul(sincl, y);
    }
    cplx excl = shfl_up(incl, 1);
    if (lane == 0) excl = {1.f, 0.f};
    cplx later = shfl_down(sincl, 1);
    if (lane == 31) later = {1.f, 0.f};
    const cplx block_total = shfl_idx(incl, 31);

    if ((n & 3) == 0 && t0 + kTokPerLane <= n) {
        // whole 16-byte units: a lane's four tokens are contiguous and 16-byte aligned
        if (a.m) *reinterpret_cast<float4 *>(a.m + base + t0) = make_float4(mm[0], mm[1], mm[2], mm[3]);
        if (a.theta_p)
            *reinterpret_cast<float4 *>(a.theta_p + base + t0) = make_float4(tp[0], tp[1], tp[2], tp[3]);
        if (a.gate) {
            float4 *gp = reinterpret_cast<float4 *>(a.gate + base + t0);
            gp[0] = make_float4(gt[0].re, gt[0].im, gt[1].re, gt[1].im);
            gp[1] = make_float4(gt[2].re, gt[2].im, gt[3].re, gt[3].im);
        }
        if (a.prefix) {
            cplx p[kTokPerLane];
#pragma unroll
            for (int k = 0; k < kTokPerLane; ++k) p[k] = cmul(excl, lp[k]);
            float4 *pp = reinterpret_cast<float4 *>(a.prefix + base + t0);
            pp[0] = make_float4(p[0].re, p[0].im, p[1].re, p[1].im);
            pp[1] = make_float4(p[2].re, p[2].im, p[3].re, p[3].im);
        }
        if (a.suffix) {
            cplx q[kTokPerLane];
#pragma unroll
            for (int k = 0; k < kTokPerLane; ++k) q[k] = cmul(ls[k], later);
            float4 *sp = reinterpret_cast<float4 *>(a.suffix + base + t0);
            sp[0] = make_float4(q[0].re, q[0].im, q[1].re, q[1].im);
            sp[1] = make_float4(q[2].re, q[2].im, q[3].re, q[3].im);
        }
    } else {
#pragma unroll
    for (int k = 0; k < kTokPerLane; ++k) {
        const int t = t0 + k;
        if (t >= n) break;
        if (a.m) a.m[base + t] = mm[k];
        if (a.theta_p) a.theta_p[base + t] = tp[k];
        if (a.gate) a.gate[base + t] = make_float2(gt[k].re, gt[k].im);
        if (a.prefix) {
            const cplx p = cmul(excl, lp[k]);
            a.prefix[base + t] = make_float2(p.re, p.im);
        }
        if (a.suffix) {
            const cplx s = cmul(ls[k], later);
            a.suffix[base + t] = make_float2(s.re, s.im);
        }
    }
    }
    if (a.carry && lane == 0)
        a.carry[bh * nb + blk] = make_float2(block_total.re, block_total.im);
}

// Finiteness scans: 16-byte loads where a head's values start on a 16-byte boundary and fill
// whole 16-byte units (the scan then runs at memory speed), one value at a time otherwise.
__global__ void check_finite_bf16_kernel(const __nv_bfloat16 *x, int64_t per_head,
                                         const __grid_constant__ HeadTable tab, int32_t *status)
{
    const int slot = blockIdx.y;
    if (slot >= tab.count) return;
    const uint16_t *p = reinterpret_cast<const uint16_t *>(x) + (int64_t)tab.bh[slot] * per_head;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, stride = (int64_t)gridDim.x * blockDim.x;
    bool bad = false;
    if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0 && (per_head & 7) == 0) {
        // eight values a load; a bf16 is inf or NaN when its exponent field (0x7F80) is all ones
        const uint4 *p4 = reinterpret_cast<const uint4 *>(p);
        uint32_t hit = 0u;
#pragma unroll 4
        for (int64_t i = t0; i < per_head / 8; i += stride) {
            const uint4 w = __ldg(p4 + i);
            hit |= __vcmpeq2(w.x & 0x7F807F80u, 0x7F807F80u) | __vcmpeq2(w.y & 0x7F807F80u, 0x7F807F80u) |
                   __vcmpeq2(w.z & 0x7F807F80u, 0x7F807F80u) | __vcmpeq2(w.w & 0x7F807F80u, 0x7F807F80u);
        }
        bad = hit != 0u;
    } else {
        for (int64_t i = t0; i < per_head; i += stride)
            bad |= (p[i] & 0x7F80u) == 0x7F80u;  // exponent all ones: inf or NaN
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(status, RS_STATUS_NONFINITE_BIT);
}

__global__ void check_finite_f32_kernel(const float *x, int64_t per_head,
                                        const __grid_constant__ HeadTable tab, int32_t *status)
{
    const int slot = blockIdx.y;
    if (slot >= tab.count) return;
    const float *p = x + (int64_t)tab.bh[slot] * per_head;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x, stride = (int64_t)gridDim.x * blockDim.x;
    bool bad = false;
    if ((reinterpret_cast<uintptr_t>(p) & 15u) == 0 && (per_head & 3) == 0) {
        const uint4 *p4 = reinterpret_cast<const uint4 *>(p);
        uint32_t hit = 0u;
#pragma unroll 4
        for (int64_t i = t0; i < per_head / 4; i += stride) {
            const uint4 w = __ldg(p4 + i);
            hit |= ((w.x & 0x7F800000u) == 0x7F800000u) | ((w.y & 0x7F800000u) == 0x7F800000u) |
                   ((w.z & 0x7F800000u) == 0x7F800000u) | ((w.w & 0x7F800000u) == 0x7F800000u);
        }
        bad = hit != 0u;
    } else {
        for (int64_t i = t0; i < per_head; i += stride) bad |= !isfinite(p[i]);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(status, RS_STATUS_NONFINITE_BIT);
}

__global__ void pad_to_bf16_kernel(const void *src, int src_is_f32, int64_t rows, int cols,
                                   __nv_bfloat16 *dst, int dst_cols, int32_t *status, int check)
{
    bool bad = false;
    const int64_t total = rows * dst_cols;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total;
         e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t r = e / dst_cols;
        const int c = (int)(e - r * dst_cols);
        float v = 0.f;
        if (c < cols) {
            v = src_is_f32 ? static_cast<const float *>(src)[r * cols + c]
                           : __bfloat162float(static_cast<const __nv_bfloat16 *>(src)[r * cols + c]);
            bad |= check && !isfinite(v);
        }
        dst[e] = __float2bfloat16_rn(v);
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) flag_status(status, RS_STATUS_NONFINITE_BIT);
}

// One thread per entry (i, j) of one head's G.
__global__ void debug_path_product_kernel(const float2 *gate, const float2 *prefix,
                                          const float2 *suffix, const float2 *carry, int n,
                                          const __grid_constant__ HeadTable tab, float2 *G)
{
    const int slot = blockIdx.z;
    if (slot >= tab.count) return;
    const int i = blockIdx.y;
    const int j = blockIdx.x * blockDim.x + threadIdx.x;
    if (j >= n) return;
    const int64_t bh = tab.bh[slot];
    const int nb = (n + kBlock - 1) / kBlock;
    const float2 *ga = gate + bh * n, *pq = prefix + bh * n, *sg = suffix + bh * n;
    const float2 *T = carry + bh * nb;
    cplx out = {0.f, 0.f};
    if (j <= i) {
        const int QB = i / kBlock, KB = j / kBlock;
        if (QB == KB) {
            // as the head kernel forms it: a row of the upper half of the block reaches a key
            // of the lower half through A_i = prod_{k=64..i} a_k, then one gate at a time
            const int b0 = QB * kBlock, il = i - b0, jl = j - b0;
            cplx Gv = {1.f, 0.f};
            int top = i;
            if (il >= kBlock / 2 && jl < kBlock / 2) {
                for (int k = b0 + kBlock / 2; k <= i; ++k) Gv = cmul(Gv, {ga[k].x, ga[k].y});
                top = b0 + kBlock / 2 - 1;
            }
            for (int jj = top - 1; jj >= j; --jj) Gv = diag_step(Gv, {ga[jj + 1].x, ga[jj + 1].y});
            out = Gv;
        } else {
            cplx C = {1.f, 0.f};
            for (int b = QB - 1; b > KB; --b) C = carry_step(C, {T[b].x, T[b].y});
            out = offdiag_product({pq[i].x, pq[i].y}, key_scale(C, {sg[j].x, sg[j].y}));
        }
    }
    G[((int64_t)slot * n + i) * n + j] = make_float2(out.re, out.im);
}

}  // namespace

cudaError_t launch_gate_prep(const GatePrepArgs &a, const HeadTable &tab, cudaStream_t s)
{
    const int nb = (a.n + kBlock - 1) / kBlock;
    const int64_t warps = (int64_t)tab.count * nb;
    const int grid = (int)((warps + 3) / 4);
    if (grid == 0) return cudaSuccess;
    gate_prep_kernel<<<grid, 128, 0, s>>>(a, tab);
    return cudaGetLastError();
}

cudaError_t launch_check_finite_bf16(const __nv_bfloat16 *x, int64_t per_head, const HeadTable &tab,
                                     int32_t *status, cudaStream_t s)
{
    if (tab.count == 0 || per_head == 0) return cudaSuccess;
    const int gx = (int)std::min<int64_t>((per_head + 256 * 32 - 1) / (256 * 32), 64);
    check_finite_bf16_kernel<<<dim3(gx, tab.count), 256, 0, s>>>(x, per_head, tab, status);
    return cudaGetLastError();
}

cudaError_t launch_check_finite_f32(const float *x, int64_t per_head, const HeadTable &tab,
                                    int32_t *status, cudaStream_t s)
{
    if (tab.count == 0 || per_head == 0) return cudaSuccess;
    const int gx = (int)std::min<int64_t>((per_head + 256 * 16 - 1) / (256 * 16), 64);
    check_finite_f32_kernel<<<dim3(gx, tab.count), 256, 0, s>>>(x, per_head, tab, status);
    return cudaGetLastError();
}

cudaError_t launch_pad_to_bf16(const void *src, int src_is_f32, int64_t rows, int cols,
                               __nv_bfloat16 *dst, int dst_cols, int32_t *status,
                               int check_finite, cudaStream_t s)
{
    const int64_t total = rows * dst_cols;
    if (total == 0) return cudaSuccess;
    const int grid = (int)std::min<int64_t>((total + 255) / 256, 152 * 16);
    pad_to_bf16_kernel<<<grid, 256, 0, s>>>(src, src_is_f32, rows, cols, dst, dst_cols, status,
                                            check_finite);
    return cudaGetLastError();
}

cudaError_t launch_debug_path_product(const float2 *gate, const float2 *prefix,
                                      const float2 *suffix, const float2 *carry, int n,
                                      const HeadTable &tab, float2 *G, cudaStream_t s)
{
    if (tab.count == 0 || n == 0) return cudaSuccess;
    debug_path_product_kernel<<<dim3((n + 127) / 128, n, tab.count), 128, 0, s>>>(
        gate, prefix, suffix, carry, n, tab, G);
    return cudaGetLastError();
}

}  // namespace rs
