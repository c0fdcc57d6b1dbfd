// operator.cu -- the materialised operator W [n, n] of each head (K4).
//
// "Resolvent Operator", section "Object": W_ij = G_ij e^{qk s_ij} / Z_i^beta with
// Z_i = sum_{j<=i} R_ij e^{qk s_ij}, evaluated in the log domain of section "Evaluation and
// refusals" (the maximum of qk s_ij over the live entries shifts the sum); the Rust API's
// `operator`. W has n^2 entries per head, so writing it is the cost: one CTA takes one
// 128-row tile of one head and makes two passes over its key tiles, each key tile's logits
// S = Q K^T computed by one tcgen05.mma into TMEM:
//   pass 1: the live maximum M_i and the shifted sum Z'_i = sum R_ij 2^{t_ij - M_i} (log2
//           units), row by row (one thread per row);
//   pass 2: W_ij = G_ij 2^{t_ij - M_i} 2^{(1-beta) M_i} Z'_i^{-beta}, written as Re and Im
//           planes, every row a contiguous 512-byte run per key tile; entries above the
//           diagonal and key tiles beyond the first exactly-zero carry are written as 0.
// G across blocks is prefix_i * C * suffix_j (C the product of the whole blocks between, the
// carry of K1); inside the diagonal tile it is formed one gate at a time from j = i down.
// Gates are only multiplied, so every structural zero of G is an exact 0 of W.
#include "head_common.cuh"

namespace rs {

namespace {

using namespace head;

template <int DP>
struct OpCfg {
    static constexpr uint32_t q_bytes = (DP / 64) * kRegion;
    static constexpr uint32_t k_bytes = (DP / 64) * kRegion;
    static constexpr uint32_t q = 0, k = q_bytes;
    static constexpr uint32_t c = k + k_bytes;        // float2 [128] c_j = C * suffix_j
    static constexpr uint32_t cm = c + 128 * 8;       // float [128] |c_j|
    static constexpr uint32_t ga = cm + 128 * 4;      // float2 [128] gates of the query block
    static constexpr uint32_t gm = ga + 128 * 8;      // float [128] |a|
    static constexpr uint32_t bars = gm + 128 * 4;    // q, k, mma
    static constexpr uint32_t misc = bars + 3 * 8;    // tmem slot, abort
    static constexpr uint32_t end = misc + 16;
    static constexpr uint32_t alloc = end + 1024;
};

template <int DP, bool GATED>
__global__ void __launch_bounds__(128)
operator_kernel(HeadArgs a, const __grid_constant__ HeadTable tab,
                const __grid_constant__ HeadMaps maps, float *W_re, float *W_im)
{
    using L = OpCfg<DP>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bar_q = reinterpret_cast<uint64_t *>(smem + L::bars);
    uint64_t *bar_k = bar_q + 1, *bar_mma = bar_q + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc);
    volatile int *s_abort = reinterpret_cast<int *>(smem + L::misc) + 1;
    float2 *s_c = reinterpret_cast<float2 *>(smem + L::c);
    float *s_cm = reinterpret_cast<float *>(smem + L::cm);
    float2 *s_ga = reinterpret_cast<float2 *>(smem + L::ga);
    float *s_gm = reinterpret_cast<float *>(smem + L::gm);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = a.n, nqt = (n + 127) / 128;
    const int QB = nqt - 1 - (int)(blockIdx.x / tab.count);
    const int slot = (int)(blockIdx.x % tab.count);
    const int bh = tab.bh[slot];
    const float beta = tab.beta[slot], qk = tab.qk[slot];
    const int64_t tok0 = (int64_t)bh * n;
    const int i = tid, row = QB * 128 + i;
    const bool valid = row < n;
    const float scale2 = qk * 1.4426950408889634f / sqrtf((float)a.d);

    if (tid == 0) {
        mbar_init(bar_q, 1);
        mbar_init(bar_k, 1);
        mbar_init(bar_mma, 1);
        *s_abort = 0;
        fence_mbar_init();
        prefetch_tmap(&maps.q);
        prefetch_tmap(&maps.k);
        mbar_arrive_expect_tx(bar_q, L::q_bytes);
        for (int rr = 0; rr < DP / 64; ++rr)
            tma_load_3d(smem + L::q + rr * kRegion, &maps.q, bar_q, rr * 64, QB * 128, bh);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, 128);
        tmem_relinquish();
    }
    cplx pq = {1.f, 0.f};
    float rq = valid ? 1.f : 0.f;
    if (GATED) {
        pq = {0.f, 0.f};
        if (valid) {
            const float2 v = a.prefix[tok0 + row];
            pq = {v.x, v.y};
            rq = cabs(pq);
        }
        float2 av = make_float2(0.f, 0.f);
        if (valid) av = a.gate[tok0 + row];
        s_ga[i] = av;
        s_gm[i] = cabs({av.x, av.y});
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);
    const float2 *Tc = a.carry + (int64_t)bh * nqt;
    constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
    const uint64_t dq = sw128_desc(sbase + L::q, 16, 1024);
    const uint64_t dk = sw128_desc(sbase + L::k, 16, 1024);
    bool ok = wait_bar(bar_q, 0, s_abort, a.status);
    uint32_t kphase = 0;

    // S = Q K(kb)^T into TMEM columns [0, 128); every thread then reads its row
    auto logits = [&](int kb) -> bool {
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_k, L::k_bytes);
            for (int rr = 0; rr < DP / 64; ++rr)
                tma_load_3d(smem + L::k + rr * kRegion, &maps.k, bar_k, rr * 64, kb * 128, bh);
        }
        bool good = wait_bar_warp(bar_k, kphase, s_abort, a.status);
        if (tid == 0 && good) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < DP / 16; ++ks) {
                const uint32_t off = ((ks >> 2) * kRegion + (ks & 3) * 32) >> 4;
                umma_bf16_ss(tmem, dq + off, dk + off, idesc_s, ks > 0 ? 1u : 0u);
            }
            umma_commit(bar_mma);
        }
        good = good && wait_bar_warp(bar_mma, kphase, s_abort, a.status);
        kphase ^= 1u;
        tc_fence_after();
        return __syncthreads_and(good) != 0;
    };
    // c_j = C * suffix_j of key tile kb, one thread per key
    auto key_scales = [&](int kb, cplx C) {
        const float2 sg = a.suffix[tok0 + kb * 128 + tid];
        const cplx c = key_scale(C, {sg.x, sg.y});
        s_c[tid] = make_float2(c.re, c.im);
        s_cm[tid] = cabs(c);
        __syncthreads();
    };
    // the key tiles that can be live: off-diagonal ones up to the first exactly-zero carry
    int numkv = QB;
    if (GATED) {
        cplx C = {1.f, 0.f};
        for (int t = 0; t < QB; ++t) {
            if (!cnonzero(C)) {
                numkv = t;
                break;
            }
            const float2 tv = Tc[QB - 1 - t];
            C = carry_step(C, {tv.x, tv.y});
        }
    }

    // ---------------------------------------------------------------- pass 1
    float M = -INFINITY, Z = 0.f, chk = 0.f;
    auto absorb = [&](float cmax, const float (&tt)[32], const float (&rr)[32]) {
        // fold 32 live logits (rr = R_ij, 0 for dead entries) into M and Z
        if (cmax > M) {
            Z *= (M == -INFINITY) ? 0.f : ex2_approx(M - cmax);
            M = cmax;
        }
        if (M == -INFINITY) return;
#pragma unroll
        for (int e = 0; e < 32; ++e) Z = fmaf(rr[e], rr[e] > 0.f ? ex2_approx(tt[e] - M) : 0.f, Z);
    };
    cplx C = {1.f, 0.f};
    for (int t = 0; ok && t < numkv; ++t) {
        const int kb = QB - 1 - t;
        if (GATED) key_scales(kb, C);
        if (!(ok = logits(kb))) break;
        for (int ch = 0; ch < 4; ++ch) {
            float sv[32], tt[32], rr[32];
            tmem_ld32f(trow + 32 * ch, sv);
            float cmax = -INFINITY;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                tt[e] = sv[e] * scale2;
                chk = fmaf(tt[e], 0.f, chk);
                rr[e] = valid ? (GATED ? rq * s_cm[32 * ch + e] : 1.f) : 0.f;
                if (rr[e] > 0.f) cmax = fmaxf(cmax, tt[e]);
            }
            absorb(cmax, tt, rr);
        }
        tc_fence_before();
        __syncthreads();  // S and the key scales are read before the next tile replaces them
        if (GATED) {
            const float2 tv = Tc[kb];
            C = carry_step(C, {tv.x, tv.y});
        }
    }
    // the diagonal tile: G_ij one gate at a time from j = i down
    if (ok && (ok = logits(QB))) {
        float R = 1.f;
        for (int ch = 3; ch >= 0; --ch) {
            float sv[32], tt[32], rr[32];
            tmem_ld32f(trow + 32 * ch, sv);
            float cmax = -INFINITY;
#pragma unroll
            for (int e = 31; e >= 0; --e) {
                const int j = 32 * ch + e;
                if (GATED && j < i) R *= s_gm[j + 1];
                tt[e] = sv[e] * scale2;
                const bool causal = valid && j <= i;
                if (causal) chk = fmaf(tt[e], 0.f, chk);
                rr[e] = causal ? R : 0.f;
                if (rr[e] > 0.f) cmax = fmaxf(cmax, tt[e]);
            }
            absorb(cmax, tt, rr);
        }
        tc_fence_before();
        __syncthreads();
    }
    bool bad = false;
    float f = 0.f;
    if (valid && ok) {
        bad = isnan(chk) || !isfinite(M) || !(Z > 0.f) || !isfinite(Z);
        f = (beta == 0.f) ? exp2f(M) : exp2f((1.f - beta) * M - beta * log2f(Z));
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(a.status, RS_STATUS_NONFINITE_BIT);

    // ---------------------------------------------------------------- pass 2
    float *wre = W_re + (tok0 + row) * (int64_t)n;
    float *wim = W_im + (tok0 + row) * (int64_t)n;
    const bool vec = (n & 3) == 0;
    // one 32-key chunk of row i at key j0 (clipped at n)
    auto put = [&](int j0, const float (&vr)[32], const float (&vi)[32]) {
        if (!valid) return;
        if (vec && j0 + 32 <= n) {
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                *reinterpret_cast<float4 *>(wre + j0 + e) = make_float4(vr[e], vr[e + 1], vr[e + 2], vr[e + 3]);
                *reinterpret_cast<float4 *>(wim + j0 + e) = make_float4(vi[e], vi[e + 1], vi[e + 2], vi[e + 3]);
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if (j0 + e < n) {
                    wre[j0 + e] = vr[e];
                    wim[j0 + e] = vi[e];
                }
        }
    };
    const cplx fpq = cmul(pq, {f, 0.f});
    C = {1.f, 0.f};
    for (int t = 0; ok && t < numkv; ++t) {
        const int kb = QB - 1 - t;
        if (GATED) key_scales(kb, C);
        if (!(ok = logits(kb))) break;
        for (int ch = 0; ch < 4; ++ch) {
            float sv[32], vr[32], vi[32];
            tmem_ld32f(trow + 32 * ch, sv);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int j = 32 * ch + e;
                const float p = ex2_approx(fmaf(sv[e], scale2, -M));
                if (GATED) {
                    const float2 c = s_c[j];
                    const bool live = rq * s_cm[j] > 0.f;
                    const cplx w = cmul(fpq, {c.x, c.y});
                    vr[e] = live ? w.re * p : 0.f;  // G = 0 exactly: W = 0 (never 0 * inf)
                    vi[e] = live ? w.im * p : 0.f;
                } else {
                    vr[e] = f * p;
                    vi[e] = 0.f;
                }
            }
            put(kb * 128 + 32 * ch, vr, vi);
        }
        tc_fence_before();
        __syncthreads();
        if (GATED) {
            const float2 tv = Tc[kb];
            C = carry_step(C, {tv.x, tv.y});
        }
    }
    if (ok && (ok = logits(QB))) {
        cplx G = {1.f, 0.f};
        float R = 1.f;
        for (int ch = 3; ch >= 0; --ch) {
            float sv[32], vr[32], vi[32];
            tmem_ld32f(trow + 32 * ch, sv);
#pragma unroll
            for (int e = 31; e >= 0; --e) {
                const int j = 32 * ch + e;
                if (GATED && j < i) {
                    const float2 an = s_ga[j + 1];
                    G = diag_step(G, {an.x, an.y});
                    R *= s_gm[j + 1];
                }
                const bool live = valid && j <= i && R > 0.f;
                const float p = live ? f * ex2_approx(fmaf(sv[e], scale2, -M)) : 0.f;
                vr[e] = GATED ? G.re * p : p;
                vi[e] = GATED ? G.im * p : 0.f;
            }
            put(QB * 128 + 32 * ch, vr, vi);
        }
        tc_fence_before();
        __syncthreads();
    }
    // zeros: key tiles past the first zero carry, and everything above the diagonal tile
    if (ok && valid) {
        float zr[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) zr[e] = 0.f;
        for (int kb = 0; kb < QB - numkv; ++kb)
            for (int ch = 0; ch < 4; ++ch) put(kb * 128 + 32 * ch, zr, zr);
        for (int j0 = (QB + 1) * 128; j0 < n; j0 += 32) put(j0, zr, zr);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 128);
    }
}

template <int DP, bool GATED>
cudaError_t launch_o(const HeadArgs &a, const HeadTable &tab, const HeadMaps &maps, float *W_re,
                     float *W_im, cudaStream_t s)
{
    using L = OpCfg<DP>;
    auto k = operator_kernel<DP, GATED>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::alloc);
    if (e != cudaSuccess) return e;
    const int nqt = (a.n + 127) / 128;
    k<<<nqt * tab.count, 128, L::alloc, s>>>(a, tab, maps, W_re, W_im);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_operator(const HeadArgs &a, const HeadTable &tab, const HeadMaps &maps, int dpad,
                            float *W_re, float *W_im, cudaStream_t s)
{
    if (tab.count == 0 || a.n == 0) return cudaSuccess;
    const bool gated = tab.g[0] != 0.f;
    if (dpad == 64)
        return gated ? launch_o<64, true>(a, tab, maps, W_re, W_im, s) : launch_o<64, false>(a, tab, maps, W_re, W_im, s);
    return gated ? launch_o<128, true>(a, tab, maps, W_re, W_im, s) : launch_o<128, false>(a, tab, maps, W_re, W_im, s);
}

}  // namespace rs
