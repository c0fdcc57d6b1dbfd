// head_fwd.cu -- the fused causal tiled resolvent head (K2) on the sm_103a tensor cores.
//
// "Resolvent Operator", section "Object": W_ij = G_ij e^{qk s_ij} / Z_i^beta and
// O_i = sum_{j<=i} W_ij V_j, evaluated in the log domain of section "Evaluation and
// refusals": the maximum of qk s_ij over the live entries (R_ij > 0) shifts the sum Z.
//
// One CTA owns one 128-row query tile QB of one head; thread i owns row i (the TMEM lane
// layout of an M = 128 accumulator). Key tiles run from KB = QB-1 down to 0, then the
// diagonal tile:
//   * TMA brings K, V (and Q once) into 128-byte-swizzled shared memory;
//   * tcgen05.mma forms S = Q K^T in TMEM (bf16 in, fp32 accumulate);
//   * each thread reads its S row, masks dead entries, keeps the running live maximum M
//     and the shifted sum Z', and writes P = 2^{t - M} (bf16) into shared memory;
//   * across blocks the path product factors as prefix_i * C * suffix_j (gate_products.cuh):
//     V_j is scaled by c_j = C suffix_j into [Re | Im] halves, so one MMA with N = 2 dv
//     accumulates sum_j P_ij c_j V_j; the row factor prefix_i multiplies the accumulator
//     once, after the last off-diagonal tile. C only ever takes more factors, so once it
//     is exactly 0 every farther tile is dead and the loop stops;
//   * the diagonal tile forms G_ij explicitly (one gate per step from j = i down) and runs
//     two MMAs, Re(P G) V and Im(P G) V;
//   * the epilogue scales by e^{(1-beta) M} Z'^{-beta}; an exact 0 stays 0.
// Heads with g = 0 have G = 1: no gate products, no V scaling, real accumulator only.
//
// Every wait on an mbarrier is bounded; one that runs out sets RS_STATUS_TIMEOUT and the
// CTA winds down (TMEM is always freed).
#include "gate_products.cuh"

namespace rs {

namespace {

constexpr int kThreads = 128;
constexpr uint32_t kRegion = 128 * 128;  // one 128-row x 128-byte swizzled region (16 KB)

template <int DP, int DVP>
struct Layout {
    static constexpr uint32_t q = 0;
    static constexpr uint32_t k = q + (DP / 64) * kRegion;
    static constexpr uint32_t vx = k + (DP / 64) * kRegion;         // V (or V'_re) then V'_im
    static constexpr uint32_t p = vx + 2 * (DVP / 64) * kRegion;     // P (or Re P on the diagonal)
    static constexpr uint32_t pim = q;                               // Im P on the diagonal: Q, K are dead by then
    static constexpr uint32_t small = p + 2 * kRegion;
    static constexpr uint32_t c = small;                             // float2 [128] key scales c_j
    static constexpr uint32_t rc = c + 128 * 8;                      // float  [128] |c_j|
    static constexpr uint32_t ga = rc + 128 * 4;                     // float2 [128] gates of the query block
    static constexpr uint32_t gm = ga + 128 * 8;                     // float  [128] |a|
    static constexpr uint32_t bars = gm + 128 * 4;                   // 2 mbarriers
    static constexpr uint32_t tmem_slot = bars + 16;
    static constexpr uint32_t bytes = tmem_slot + 16;
    static constexpr uint32_t alloc = bytes + 1024;                  // slack for 1024-byte alignment
    static constexpr uint32_t acc_cols = 2 * DVP;
    static constexpr uint32_t s_col = acc_cols;
    static constexpr uint32_t tmem_cols = (acc_cols + 128 <= 256) ? 256 : 512;
};

__device__ __forceinline__ void store_p_chunk(uint32_t base, int row, int chunk16, uint4 v)
{
    // chunk16: which 8-key chunk (0..15) of the 128 keys
    const int region = chunk16 >> 3, c = chunk16 & 7;
    const uint32_t addr = base + region * kRegion + row * 128 + ((c ^ (row & 7)) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t addr)
{
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr));
    return v;
}

__device__ __forceinline__ void sts128(uint32_t addr, uint4 v)
{
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// Multiplies this thread's accumulator row (ncols fp32 columns from `col`) by alpha.
__device__ __forceinline__ void scale_acc_row(uint32_t trow, int ncols, float alpha)
{
    for (int cc = 0; cc < ncols; cc += 32) {
        uint32_t r[32];
        RS_TMEM_LD32(trow + cc, r);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
        RS_TMEM_ST32(trow + cc, r);
    }
    tmem_st_wait();
}

// Complex row factor: acc_re + i acc_im <- z * (acc_re + i acc_im).
__device__ __forceinline__ void cscale_acc_row(uint32_t trow, int dvp, cplx z)
{
    for (int cc = 0; cc < dvp; cc += 32) {
        uint32_t re[32], im[32];
        RS_TMEM_LD32(trow + cc, re);
        RS_TMEM_LD32(trow + dvp + cc, im);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const cplx x = cmul(z, {__uint_as_float(re[e]), __uint_as_float(im[e])});
            re[e] = __float_as_uint(x.re);
            im[e] = __float_as_uint(x.im);
        }
        RS_TMEM_ST32(trow + cc, re);
        RS_TMEM_ST32(trow + dvp + cc, im);
    }
    tmem_st_wait();
}

template <int DP, int DVP>
__global__ void __launch_bounds__(kThreads, 1)
head_fwd_kernel(HeadArgs a, const __grid_constant__ HeadTable tab,
                const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                const __grid_constant__ CUtensorMap tv)
{
    using L = Layout<DP, DVP>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bar_tma = reinterpret_cast<uint64_t *>(smem + L::bars);
    uint64_t *bar_mma = bar_tma + 1;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::tmem_slot);
    float2 *s_c = reinterpret_cast<float2 *>(smem + L::c);
    float *s_rc = reinterpret_cast<float *>(smem + L::rc);
    float2 *s_ga = reinterpret_cast<float2 *>(smem + L::ga);
    float *s_gm = reinterpret_cast<float *>(smem + L::gm);

    const int tid = threadIdx.x, warp = tid >> 5;
    const int n = a.n;
    const int nqt = (n + 127) / 128;
    const int QB = nqt - 1 - (int)(blockIdx.x / tab.count);
    const int slot = (int)(blockIdx.x % tab.count);
    const int bh = tab.bh[slot];
    const float beta = tab.beta[slot], qk = tab.qk[slot], g = tab.g[slot];
    const bool gated = g != 0.f;
    const bool qk_on = qk != 0.f;
    const int sQ = QB * 128;
    const int row = sQ + tid;
    const bool valid = row < n;
    const int64_t tok0 = (int64_t)bh * n;

    if (tid == 0) {
        mbar_init(bar_tma, 1);
        mbar_init(bar_mma, 1);
        fence_mbar_init();
        prefetch_tmap(&tq);
        prefetch_tmap(&tk);
        prefetch_tmap(&tv);
    }
    if (warp == 0) {
        tmem_alloc(tmem_slot, L::tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t trow = tmem + ((uint32_t)(warp * 32) << 16);  // this warp's TMEM lanes
    const uint32_t t_acc = tmem, t_s = tmem + L::s_col;

    const float scale2 = qk * 1.4426950408889634f / sqrtf((float)a.d);  // qk log2(e) / sqrt(d)
    const uint32_t kv_bytes = (DP / 64 + DVP / 64) * kRegion;             // K and V tiles
    const uint32_t q_bytes = (DP / 64) * kRegion;
    constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
    constexpr uint32_t idesc_pv_real = idesc_bf16(128, DVP, false, true);
    constexpr uint32_t idesc_pv_cplx = idesc_bf16(128, 2 * DVP, false, true);

    uint32_t ph_tma = 0, ph_mma = 0;
    bool ok = true;           // no wait has run out (uniform: every thread waits on the same barriers)
    bool q_loaded = false;
    bool acc_started = false;

    // row state
    cplx pq = {0.f, 0.f};
    float rq = 0.f;
    if (gated && valid) {
        const float2 v = a.prefix[tok0 + row];
        pq = {v.x, v.y};
        rq = cabs(pq);
    } else if (valid) {
        pq = {1.f, 0.f};  // ungated: every gate is 1
        rq = 1.f;
    }
    float M2 = -INFINITY;  // running live maximum of qk s log2(e)
    float Zs = 0.f;        // sum of R 2^{t - M}
    float chk = 0.f;       // becomes NaN if any evaluated logit is not finite

    auto load_tiles = [&](int kb) {
        if (tid == 0) {
            mbar_arrive_expect_tx(bar_tma, kv_bytes + (q_loaded ? 0u : q_bytes));
            if (!q_loaded)
                for (int r = 0; r < DP / 64; ++r)
                    tma_load_3d(smem + L::q + r * kRegion, &tq, bar_tma, r * 64, sQ, bh);
            for (int r = 0; r < DP / 64; ++r)
                tma_load_3d(smem + L::k + r * kRegion, &tk, bar_tma, r * 64, kb * 128, bh);
            for (int r = 0; r < DVP / 64; ++r)
                tma_load_3d(smem + L::vx + r * kRegion, &tv, bar_tma, r * 64, kb * 128, bh);
        }
        q_loaded = true;
    };
    // Waits are bounded; `ok` turns false when one runs out. It is made uniform across the
    // CTA (__syncthreads_and) before any decision that changes control flow.
    auto wait_tma = [&]() {
        ok = __all_sync(0xffffffffu, ok && mbar_wait(bar_tma, ph_tma, kWaitLimitNs));
        ph_tma ^= 1;
    };
    auto wait_mma = [&]() {
        ok = __all_sync(0xffffffffu, ok && mbar_wait(bar_mma, ph_mma, kWaitLimitNs));
        ph_mma ^= 1;
        tc_fence_after();
    };
    auto issue_s = [&]() {
        if (tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < DP / 16; ++ks) {
                const uint32_t off = (ks >> 2) * kRegion + (ks & 3) * 32;
                umma_bf16_ss(t_s, sw128_desc(sbase + L::q + off, 16, 1024),
                             sw128_desc(sbase + L::k + off, 16, 1024), idesc_s, ks > 0);
            }
            umma_commit(bar_mma);
        }
    };
    auto load_s_row = [&](float (&s)[128]) {
#pragma unroll
        for (int cc = 0; cc < 128; cc += 32) {
            uint32_t r[32];
            RS_TMEM_LD32(trow + L::s_col + cc, r);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 32; ++e) s[cc + e] = __uint_as_float(r[e]);
        }
    };

    // -------------------------------------------------------------- off-diagonal tiles
    const int rows_alive = __syncthreads_or(valid && (!gated || rq > 0.f));
    cplx C = {1.f, 0.f};
    for (int KB = QB - 1; KB >= 0 && rows_alive && ok; --KB) {
        if (gated && !cnonzero(C)) break;  // every farther key tile is exactly dead
        load_tiles(KB);
        if (gated) {
            const float2 sg = a.suffix[tok0 + KB * 128 + tid];
            const cplx c = key_scale(C, {sg.x, sg.y});
            s_c[tid] = make_float2(c.re, c.im);
            s_rc[tid] = cabs(c);
        }
        wait_tma();
        ok = __syncthreads_and(ok);
        if (!ok) break;

        float s[128];
        if (qk_on) {
            issue_s();
            wait_mma();
            load_s_row(s);
        } else {
#pragma unroll
            for (int j = 0; j < 128; ++j) s[j] = 0.f;
        }

        // live maximum of this tile
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < 128; j += 4) {
            const float4 w = gated ? *reinterpret_cast<const float4 *>(s_rc + j)
                                   : make_float4(1.f, 1.f, 1.f, 1.f);
            const float wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float t2 = s[j + e] * scale2;
                s[j + e] = t2;
                chk = fmaf(t2, 0.f, chk);
                const bool live = valid && rq * wv[e] > 0.f;
                mt = live ? fmaxf(mt, t2) : mt;
            }
        }
        const float mnew = fmaxf(M2, mt);
        float alpha = 1.f;
        if (mnew > M2) {
            alpha = (M2 == -INFINITY) ? 0.f : ex2_approx(M2 - mnew);
            Zs *= alpha;
            M2 = mnew;
        }
        if (__any_sync(0xffffffffu, acc_started && alpha != 1.f))
            scale_acc_row(trow, gated ? 2 * DVP : DVP, acc_started ? alpha : 1.f);

        // P = 2^{t - M} on live entries, Z' += |c_j| P
#pragma unroll
        for (int j = 0; j < 128; j += 8) {
            const float4 w0 = gated ? *reinterpret_cast<const float4 *>(s_rc + j)
                                    : make_float4(1.f, 1.f, 1.f, 1.f);
            const float4 w1 = gated ? *reinterpret_cast<const float4 *>(s_rc + j + 4)
                                    : make_float4(1.f, 1.f, 1.f, 1.f);
            const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
            float p[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                const bool live = valid && rq * wv[e] > 0.f;
                p[e] = live ? ex2_approx(s[j + e] - M2) : 0.f;
                Zs = fmaf(wv[e], p[e], Zs);
            }
            store_p_chunk(sbase + L::p, tid, j >> 3,
                          make_uint4(pack_bf16x2(p[0], p[1]), pack_bf16x2(p[2], p[3]),
                                     pack_bf16x2(p[4], p[5]), pack_bf16x2(p[6], p[7])));
        }

        // V'_j = c_j V_j: Re in place, Im into the second half (thread = key row)
        if (gated) {
            const float2 c = s_c[tid];
#pragma unroll
            for (int r = 0; r < DVP / 64; ++r) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    const uint32_t addr = sbase + L::vx + r * kRegion + tid * 128 + ch * 16;
                    const uint4 v = lds128(addr);
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    uint32_t ore[4], oim[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float2 f = unpack_bf16x2(w[e]);
                        ore[e] = pack_bf16x2(f.x * c.x, f.y * c.x);
                        oim[e] = pack_bf16x2(f.x * c.y, f.y * c.y);
                    }
                    sts128(addr, make_uint4(ore[0], ore[1], ore[2], ore[3]));
                    sts128(addr + (DVP / 64) * kRegion, make_uint4(oim[0], oim[1], oim[2], oim[3]));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok);
        if (!ok) break;
        if (tid == 0) {
            tc_fence_after();
            const uint32_t idesc = gated ? idesc_pv_cplx : idesc_pv_real;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t aoff = (ks >> 2) * kRegion + (ks & 3) * 32;
                umma_bf16_ss(t_acc, sw128_desc(sbase + L::p + aoff, 16, 1024),
                             sw128_desc(sbase + L::vx + ks * 2048, kRegion, 1024), idesc,
                             (acc_started || ks > 0) ? 1u : 0u);
            }
            umma_commit(bar_mma);
        }
        wait_mma();
        acc_started = true;
        if (gated) {
            const float2 T = a.carry[(int64_t)bh * nqt + KB];
            C = carry_step(C, {T.x, T.y});
        }
    }

    ok = __syncthreads_and(ok);

    // -------------------------------------------------------------- row factor prefix_i
    if (ok && gated && acc_started) {
        cscale_acc_row(trow, DVP, pq);
        Zs *= rq;
    }

    // -------------------------------------------------------------- diagonal tile
    if (ok) {
        load_tiles(QB);
        if (gated) {
            float2 av = make_float2(0.f, 0.f);
            if (valid) av = a.gate[tok0 + row];
            s_ga[tid] = av;
            s_gm[tid] = cabs({av.x, av.y});
        }
        wait_tma();
    }
    ok = __syncthreads_and(ok);
    if (ok) {
        float s[128];
        if (qk_on) {
            issue_s();
            wait_mma();
            load_s_row(s);
        } else {
#pragma unroll
            for (int j = 0; j < 128; ++j) s[j] = 0.f;
        }
        const int i = tid;
        // pass 1: causal logits, the live maximum
        float mt = -INFINITY;
        {
            cplx G = {1.f, 0.f};
            float R = 1.f;
#pragma unroll
            for (int j = 127; j >= 0; --j) {
                if (gated && j < i) {
                    const float2 an = s_ga[j + 1];
                    G = diag_step(G, {an.x, an.y});
                    R *= s_gm[j + 1];
                }
                const float t2 = s[j] * scale2;
                s[j] = t2;
                const bool causal = valid && j <= i;
                if (causal) chk = fmaf(t2, 0.f, chk);
                const bool live = causal && R > 0.f;
                mt = live ? fmaxf(mt, t2) : mt;
            }
        }
        const float mnew = fmaxf(M2, mt);
        float alpha = 1.f;
        if (mnew > M2) {
            alpha = (M2 == -INFINITY) ? 0.f : ex2_approx(M2 - mnew);
            Zs *= alpha;
            M2 = mnew;
        }
        if (__any_sync(0xffffffffu, acc_started && alpha != 1.f))
            scale_acc_row(trow, gated ? 2 * DVP : DVP, acc_started ? alpha : 1.f);

        // pass 2: P G (Re into the P buffer, Im into the dead Q/K buffer)
        {
            cplx G = {1.f, 0.f};
            float R = 1.f;
            float pre[8], pim[8];
#pragma unroll
            for (int j = 127; j >= 0; --j) {
                if (gated && j < i) {
                    const float2 an = s_ga[j + 1];
                    G = diag_step(G, {an.x, an.y});
                    R *= s_gm[j + 1];
                }
                const bool live = valid && j <= i && R > 0.f;
                const float p = live ? ex2_approx(s[j] - M2) : 0.f;
                Zs = fmaf(R, p, Zs);
                pre[j & 7] = gated ? G.re * p : p;
                pim[j & 7] = G.im * p;
                if ((j & 7) == 0) {
                    store_p_chunk(sbase + L::p, tid, j >> 3,
                                  make_uint4(pack_bf16x2(pre[0], pre[1]), pack_bf16x2(pre[2], pre[3]),
                                             pack_bf16x2(pre[4], pre[5]), pack_bf16x2(pre[6], pre[7])));
                    if (gated)
                        store_p_chunk(sbase + L::pim, tid, j >> 3,
                                      make_uint4(pack_bf16x2(pim[0], pim[1]), pack_bf16x2(pim[2], pim[3]),
                                                 pack_bf16x2(pim[4], pim[5]), pack_bf16x2(pim[6], pim[7])));
                }
            }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        ok = __syncthreads_and(ok);
        if (ok && tid == 0) {
            tc_fence_after();
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
                const uint32_t aoff = (ks >> 2) * kRegion + (ks & 3) * 32;
                const uint64_t bdesc = sw128_desc(sbase + L::vx + ks * 2048, kRegion, 1024);
                umma_bf16_ss(t_acc, sw128_desc(sbase + L::p + aoff, 16, 1024), bdesc, idesc_pv_real,
                             (acc_started || ks > 0) ? 1u : 0u);
                if (gated)
                    umma_bf16_ss(t_acc + DVP, sw128_desc(sbase + L::pim + aoff, 16, 1024), bdesc,
                                 idesc_pv_real, (acc_started || ks > 0) ? 1u : 0u);
            }
            umma_commit(bar_mma);
        }
        if (ok) wait_mma();
        acc_started = true;
    }
    ok = __syncthreads_and(ok);

    // -------------------------------------------------------------- epilogue
    if (ok) {
        bool bad = false;
        float f = 0.f;
        if (valid) {
            bad = isnan(chk) || !isfinite(M2) || !(Zs > 0.f) || !isfinite(Zs);
            // O = acc e^{(1-beta) M} Z'^{-beta}, in base 2; beta log Z' is 0 at beta = 0
            f = (beta == 0.f) ? exp2f(M2) : exp2f((1.f - beta) * M2 - beta * log2f(Zs));
        }
        if (__any_sync(0xffffffffu, bad) && (tid & 31) == 0) flag_status(a.status, RS_STATUS_NONFINITE_BIT);
        float *ore = a.O_re + (tok0 + row) * (int64_t)a.dv;
        float *oim = a.O_im + (tok0 + row) * (int64_t)a.dv;
        for (int cc = 0; cc < DVP; cc += 32) {
            uint32_t re[32], im[32];
            RS_TMEM_LD32(trow + cc, re);
            if (gated) RS_TMEM_LD32(trow + DVP + cc, im);
            tmem_ld_wait();
            if (valid) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int col = cc + e;
                    if (col < a.dv) {
                        const float xr = __uint_as_float(re[e]);
                        const float xi = gated ? __uint_as_float(im[e]) : 0.f;
                        ore[col] = (xr == 0.f) ? 0.f : xr * f;  // an exact 0 stays 0 (never 0 * inf)
                        oim[col] = (xi == 0.f) ? 0.f : xi * f;
                    }
                }
            }
        }
    } else if (tid == 0) {
        flag_status(a.status, RS_STATUS_TIMEOUT_BIT);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, L::tmem_cols);
    }
}

template <int DP, int DVP>
cudaError_t launch_t(const HeadArgs &a, const HeadTable &tab, const CUtensorMap &tq,
                     const CUtensorMap &tk, const CUtensorMap &tv, cudaStream_t s)
{
    using L = Layout<DP, DVP>;
    auto k = head_fwd_kernel<DP, DVP>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::alloc);
    if (e != cudaSuccess) return e;
    const int nqt = (a.n + 127) / 128;
    k<<<nqt * tab.count, kThreads, L::alloc, s>>>(a, tab, tq, tk, tv);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_head_fwd(const HeadArgs &a, const HeadTable &tab, const CUtensorMap &tq,
                            const CUtensorMap &tk, const CUtensorMap &tv, int dpad, int dvpad,
                            cudaStream_t s)
{
    if (tab.count == 0 || a.n == 0) return cudaSuccess;
    if (dpad == 64 && dvpad == 64) return launch_t<64, 64>(a, tab, tq, tk, tv, s);
    if (dpad == 64 && dvpad == 128) return launch_t<64, 128>(a, tab, tq, tk, tv, s);
    if (dpad == 128 && dvpad == 64) return launch_t<128, 64>(a, tab, tq, tk, tv, s);
    return launch_t<128, 128>(a, tab, tq, tk, tv, s);
}

}  // namespace rs
