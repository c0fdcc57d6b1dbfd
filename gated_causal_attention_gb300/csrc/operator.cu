// operator.cu -- the materialised operator W [n, n] of each head (K4).
//
// "Resolvent Operator", section "Object": W_ij = G_ij e^{qk s_ij} / Z_i^beta with
// Z_i = sum_{j<=i} R_ij e^{qk s_ij}, evaluated in the log domain of section "Evaluation and
// refusals" (the maximum of qk s_ij over the live entries shifts the sum); the Rust API's
// `operator`. Writing W (n^2 complex entries per head) is the whole cost, so the work is cut
// in two launches that both spread evenly over the SMs:
//   row statistics -- units of (head, 128-row query tile, a run of CH key tiles); each unit
//       folds its live logits into a partial (M, Z') per row (log2 units: M the live maximum,
//       Z' = sum R_ij 2^{t_ij - M}) and records the carry product C(QB, KB) of every key
//       tile it visits;
//   write -- every 128 x 128 tile of W, lower and upper, dealt round-robin to persistent
//       CTAs; a lower tile merges its row partials, forms
//       W_ij = G_ij 2^{t_ij - M_i} 2^{(1-beta) M_i} Z'_i^{-beta} and leaves through shared
//       staging and tensor-map stores (32 x 32 swizzled blocks); tiles above the diagonal and
//       beyond an exactly-zero carry are stored from a block of zeros.
// In both, warp 8 produces: it gathers the tile's column data (the key scales C * suffix_j,
// or the gates of the diagonal block) and row data into shared memory, loads Q and K by TMA
// and issues S = Q K^T (one tcgen05.mma chain) into one of two TMEM buffers. Warps 0-7
// consume: warp w reads TMEM lanes 32 (w % 4) .. +31 (its rows) and columns 64 (w / 4) .. +63.
// G across blocks is prefix_i * C * suffix_j (C the product of the whole blocks between, the
// carry of K1); inside the diagonal tile it is formed one gate at a time from j = i down, the
// lower column half first walking the upper half's gates without writing. Both launches take
// every live/dead decision from the same values by the same operations, and the write clamps
// the exponent at 0, so an entry left out of the row maximum can never overflow. Gates are
// only multiplied, so every structural zero of G is an exact 0 of W.
#include "head_common.cuh"

namespace rs {

namespace {

using namespace head;

constexpr int kOpThreads = 288;  // warps 0-7 consume, warp 8 produces
constexpr int kProdWarp = 8;
constexpr int kConsumers = 256;
enum : int { kTileZero = 0, kTileOff = 1, kTileDiag = 2 };

template <int N>
__device__ __forceinline__ void bulk_wait_read()
{
    asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// (M, Z) <- the merge of two partial row statistics in log2 units (M = -inf: empty; a NaN
// maximum stays NaN).
__device__ __forceinline__ void merge_stats(float &M, float &Z, float M2, float Z2)
{
    if (isnan(M2)) {
        M = M2;
        return;
    }
    if (M2 == -INFINITY || isnan(M)) return;
    if (M2 > M) {
        Z = (M == -INFINITY ? 0.f : Z * exp2f(M - M2)) + Z2;
        M = M2;
    } else {
        Z += Z2 * exp2f(M2 - M);
    }
}

template <int DP, bool STATS>
struct OpLayout {
    static constexpr uint32_t qk_bytes = 2 * (DP / 64) * kRegion;  // Q and K of one stage
    static constexpr int nslot = STATS ? 0 : (DP == 64 ? 2 : 1);   // staging slots per warp
    static constexpr uint32_t stage = 0;                            // [2] stages of Q, K
    static constexpr uint32_t staging = stage + 2 * qk_bytes;       // [8][nslot] x (Re 4K, Im 4K)
    static constexpr uint32_t zero = staging + 8 * nslot * 8192;    // 4 KB of zeros (write)
    static constexpr uint32_t col = zero + (STATS ? 0 : 4096);      // float4 [2][128]
    static constexpr uint32_t colm = col + 2 * 128 * 16;            // float [2][128]
    static constexpr uint32_t rows = colm + 2 * 128 * 4;            // float4 [2][128]
    static constexpr uint32_t rq = rows + 2 * 128 * 16;             // float [2][128]
    static constexpr uint32_t xchg = rq + 2 * 128 * 4;              // float4 [2][128] (stats)
    static constexpr uint32_t kind = xchg + 2 * 128 * 16;           // int [2], then float [2] cmin
    static constexpr uint32_t bars = kind + 16;                     // kfull[2] sfull[2] sempty[2] drain
    static constexpr uint32_t misc = bars + 7 * 8;                  // tmem slot, abort flag
    static constexpr uint32_t end = misc + 16;
    static constexpr uint32_t alloc = end + 1024;
    static_assert(alloc <= 227 * 1024, "shared memory");
};

// Shared state of one CTA of either launch.
struct OpSmem {
    unsigned char *base;
    uint32_t sbase;
    float4 *col;  // (re, im, -im, re) of a key scale or a gate
    float *colm;  // its magnitude
    float4 *rows;
    float *rq;
    float4 *xchg;
    volatile int *kind;
    volatile float *cmin;  // the smallest key-scale magnitude of the tile (off-diagonal tiles)
    uint64_t *kfull, *sfull, *sempty;
    uint64_t *drain;  // the producer's own wait for its MMAs when it winds down
    uint32_t *tmem_slot;
    volatile int *abort;
};

template <class L>
__device__ __forceinline__ OpSmem op_smem(unsigned char *smem_raw)
{
    OpSmem m;
    m.base = reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    m.sbase = smem_u32(m.base);
    m.col = reinterpret_cast<float4 *>(m.base + L::col);
    m.colm = reinterpret_cast<float *>(m.base + L::colm);
    m.rows = reinterpret_cast<float4 *>(m.base + L::rows);
    m.rq = reinterpret_cast<float *>(m.base + L::rq);
    m.xchg = reinterpret_cast<float4 *>(m.base + L::xchg);
    m.kind = reinterpret_cast<volatile int *>(m.base + L::kind);
    m.cmin = reinterpret_cast<volatile float *>(m.base + L::kind + 8);
    m.kfull = reinterpret_cast<uint64_t *>(m.base + L::bars);
    m.sfull = m.kfull + 2;
    m.sempty = m.kfull + 4;
    m.drain = m.kfull + 6;
    m.tmem_slot = reinterpret_cast<uint32_t *>(m.base + L::misc);
    m.abort = reinterpret_cast<volatile int *>(m.base + L::misc) + 1;
    return m;
}

// Barriers, the TMEM buffers (2 x 128 columns) and, for the write launch, the block of zeros.
template <class L, bool ZERO_BLOCK>
__device__ __forceinline__ uint32_t op_setup(const OpSmem &m, const OpMaps &maps)
{
    const int tid = threadIdx.x, warp = tid >> 5;
    if (ZERO_BLOCK) {
        for (int e = tid; e < 1024; e += kOpThreads) reinterpret_cast<float *>(m.base + L::zero)[e] = 0.f;
        fence_proxy_async_smem();
    }
    if (tid == 0) {
        for (int b = 0; b < 2; ++b) {
            mbar_init(m.kfull + b, 1);
            mbar_init(m.sfull + b, 2);  // the producer's release of the smem data + the MMA commit
            mbar_init(m.sempty + b, 8);
        }
        mbar_init(m.drain, 1);
        *m.abort = 0;
        fence_mbar_init();
    }
    if (warp == kProdWarp && (tid & 31) == 0) {
        prefetch_tmap(&maps.q);
        prefetch_tmap(&maps.k);
    }
    if (warp == 0) {
        tmem_alloc(m.tmem_slot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    return *m.tmem_slot;
}

__device__ __forceinline__ void op_teardown(const OpSmem &m, uint32_t tmem)
{
    // the producer lane issued every MMA of the CTA: they end before TMEM is freed
    if ((threadIdx.x >> 5) == kProdWarp && (threadIdx.x & 31) == 0) drain_mma(m.drain);
    tc_fence_before();
    __syncthreads();
    if ((threadIdx.x >> 5) == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

// Global data of one lower tile, loaded into registers a tile ahead of its use so that the
// loads overlap the producer's wait for the tile's buffer.
struct TileFetch {
    float2 v[4];   // per column j = lane + 32 e: suffix_j (off-diagonal) or the block's gates
    float4 rf[4];  // per row r = lane + 32 e: write: (M, f, f prefix_r); stats: prefix_r
    float rq[4];   // write: |prefix_r|
    float2 ct;     // write: C(QB, KB); stats: the block total folded into C after the tile
    float2 wv;     // stats, first tile of a unit: block total QB - 1 - lane of the walk to it
};

template <bool GATED>
__device__ __forceinline__ void fetch_cols(const OpArgs &a, int64_t tok0, int QB, int kk, TileFetch &f)
{
    const int lane = threadIdx.x & 31, KB = QB - kk;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int j = lane + 32 * e;
        f.v[e] = make_float2(0.f, 0.f);
        if (GATED) {
            if (kk > 0) f.v[e] = a.suffix[tok0 + KB * 128 + j];
            else if (QB * 128 + j < a.n) f.v[e] = a.gate[tok0 + QB * 128 + j];
        }
    }
}

// The producer's part of lower tile number k of this CTA (KB = QB - kk <= QB), into buffer
// b = k & 1, from the tile's prefetched data f: the loads of Q and K by TMA go out first, then
// column data, row data (`rowdata(f, b)`) and kind are written, then S = Q K^T goes into TMEM
// columns [128 b, 128 b + 128). Returns false after a timeout.
template <int DP, bool GATED, class L, class RowData>
__device__ __forceinline__ bool produce_tile(const OpArgs &a, const OpMaps &maps, const OpSmem &m,
                                             uint32_t tmem, int bh, int QB, int kk, cplx C, int k,
                                             uint32_t &kph, const TileFetch &f, RowData rowdata,
                                             int withhold)
{
    const int lane = threadIdx.x & 31, b = k & 1;
    const int KB = QB - kk;
    // buffer b was last used by tile k - 2: its consumers are done with it, and so is its MMA
    if (k >= 2 && !wait_bar_warp(m.sempty + b, ((k >> 1) + 1) & 1, m.abort, a.status, 0)) return false;
    const int kind = kk == 0 ? kTileDiag : ((GATED && !cnonzero(C)) ? kTileZero : kTileOff);
    unsigned char *st = m.base + L::stage + b * L::qk_bytes;
    // test knob: block `withhold` loads nothing for its second tile, so the wait below runs out
    if (lane == 0 && kind != kTileZero && !(k == 1 && (int)blockIdx.x == withhold)) {
        mbar_arrive_expect_tx(m.kfull + b, L::qk_bytes);
        for (int rr = 0; rr < DP / 64; ++rr) {
            tma_load_3d(st + rr * kRegion, &maps.q, m.kfull + b, rr * 64, QB * 128, bh);
            tma_load_3d(st + (DP / 64 + rr) * kRegion, &maps.k, m.kfull + b, rr * 64, KB * 128, bh);
        }
    }
    if (GATED && kind != kTileZero) {
        float cmin = INFINITY;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int j = lane + 32 * e;
            const cplx c = kind == kTileOff ? key_scale(C, {f.v[e].x, f.v[e].y}) : cplx{f.v[e].x, f.v[e].y};
            const float cm = cabs(c);
            m.col[b * 128 + j] = make_float4(c.re, c.im, -c.im, c.re);
            m.colm[b * 128 + j] = cm;
            cmin = fminf(cmin, cm);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) cmin = fminf(cmin, __shfl_xor_sync(0xffffffffu, cmin, o));
        if (lane == 0) m.cmin[b] = cmin;
    }
    if (kind != kTileZero) rowdata(f, b);
    if (lane == 0) m.kind[b] = kind;
    __syncwarp();
    bool ok = true;
    if (lane == 0) {
        mbar_arrive(m.sfull + b);  // releases the column / row data written above
        if (kind == kTileZero) {
            mbar_arrive(m.sfull + b);
        } else {
            ok = wait_bar(m.kfull + b, (kph >> b) & 1u, m.abort, a.status);
            // the loads of this tile are the only ones in flight: after a timeout they still
            // land before the CTA exits
            if (!ok) mbar_wait(m.kfull + b, (kph >> b) & 1u, kDrainLimitNs);
            if (ok) {
                tc_fence_after();
                constexpr uint32_t idesc = idesc_bf16(128, 128, false, false);
                const uint32_t sq = smem_u32(st), sk = sq + (DP / 64) * kRegion;
                const uint64_t dq = sw128_desc(sq, 16, 1024), dk = sw128_desc(sk, 16, 1024);
#pragma unroll
                for (int ks = 0; ks < DP / 16; ++ks) {
                    const uint32_t off = ((ks >> 2) * kRegion + (ks & 3) * 32) >> 4;
                    umma_bf16_ss(tmem + b * 128, dq + off, dk + off, idesc, ks > 0 ? 1u : 0u);
                }
                umma_commit(m.sfull + b);
            }
        }
    }
    if (kind != kTileZero) kph ^= 1u << b;
    return __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
}

// Folds 32 logits (tt, log2 units) with weights rr (R_ij; 0 = dead) into (M, Z).
__device__ __forceinline__ void absorb32(float &M, float &Z, const float (&tt)[32], const float (&rr)[32])
{
    float cmax = -INFINITY;
#pragma unroll
    for (int e = 0; e < 32; ++e)
        if (rr[e] > 0.f) cmax = fmaxf(cmax, tt[e]);
    if (cmax > M) {
        Z = (M == -INFINITY) ? 0.f : Z * ex2_approx(M - cmax);
        M = cmax;
    }
    if (M == -INFINITY) return;
#pragma unroll
    for (int e = 0; e < 32; ++e) Z = fmaf(rr[e], rr[e] > 0.f ? ex2_approx(tt[e] - M) : 0.f, Z);
}

// ================================================================ row statistics

// Stats units of one head, chunk-major: chunk c (key tiles kk in [c CH, c CH + CH)) of every
// query tile QB >= c CH.
__device__ __forceinline__ void stats_unit(int idx, int nqt, int CH, int &QB, int &c)
{
    c = 0;
    while (idx >= nqt - c * CH) {
        idx -= nqt - c * CH;
        ++c;
    }
    QB = c * CH + idx;
}

template <int DP, bool GATED>
__global__ void __launch_bounds__(kOpThreads, 2)
operator_stats_kernel(OpArgs a, const __grid_constant__ HeadTable tab, const __grid_constant__ OpMaps maps)
{
    using L = OpLayout<DP, true>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const OpSmem m = op_smem<L>(smem_raw);
    const uint32_t tmem = op_setup<L, false>(m, maps);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = a.n, nqt = (n + 127) / 128, CH = a.chunk, NCH = (nqt + CH - 1) / CH;
    int per_head = 0;
    for (int c = 0; c < NCH; ++c) per_head += nqt - c * CH;
    const int units = per_head * tab.count;

    if (warp == kProdWarp) {
        // the CTA's (unit, tile) sequence, each tile's global data fetched one tile ahead
        struct Item {
            int u, slot, QB, c, kk;
        };
        auto locate = [&](int u, Item &it) {
            it.u = u;
            it.slot = u / per_head;
            stats_unit(u - it.slot * per_head, nqt, CH, it.QB, it.c);
            it.kk = it.c * CH;
        };
        auto fetch = [&](const Item &it, TileFetch &f) {
            const int bh = tab.bh[it.slot];
            const int64_t tok0 = (int64_t)bh * n;
            const float2 *Tc = a.carry + (int64_t)bh * nqt;
            fetch_cols<GATED>(a, tok0, it.QB, it.kk, f);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = it.QB * 128 + lane + 32 * e;
                f.rf[e] = make_float4(row < n ? 1.f : 0.f, 0.f, 0.f, 0.f);
                if (GATED && row < n) {
                    const float2 p = a.prefix[tok0 + row];
                    f.rf[e] = make_float4(p.x, p.y, 0.f, 0.f);
                }
            }
            f.ct = make_float2(1.f, 0.f);
            f.wv = make_float2(1.f, 0.f);
            if (GATED) {
                if (it.kk >= 1) f.ct = Tc[it.QB - it.kk];
                if (it.kk == it.c * CH && lane < min(32, it.kk - 1)) f.wv = Tc[it.QB - 1 - lane];
            }
        };
        auto advance = [&](Item &it) {
            if (++it.kk < min(it.c * CH + CH, it.QB + 1)) return;
            if (it.u + (int)gridDim.x < units) locate(it.u + gridDim.x, it);
            else it.u = units;
        };
        auto rowdata = [&](const TileFetch &f, int b) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
                m.rq[b * 128 + lane + 32 * e] = GATED ? cabs({f.rf[e].x, f.rf[e].y}) : f.rf[e].x;
        };
        uint32_t kph = 0;
        bool ok = true;
        Item it;
        TileFetch fn;
        if ((int)blockIdx.x < units) {
            locate(blockIdx.x, it);
            fetch(it, fn);
        } else {
            it.u = units;
        }
        cplx C = {1.f, 0.f};
        for (int k = 0; ok && it.u < units; ++k) {
            const Item cur = it;
            const TileFetch fc = fn;
            advance(it);
            if (it.u < units) fetch(it, fn);
            const int bh = tab.bh[cur.slot];
            if (GATED && cur.kk == cur.c * CH) {
                // C(QB, QB - kk): 1 at kk = 1, then one more block total per step; the walk to
                // the unit's first tile takes the prefetched totals, 32 at a time
                const float2 *Tc = a.carry + (int64_t)bh * nqt;
                C = {1.f, 0.f};
                for (int base = 1; base < cur.kk; base += 32) {
                    const int cnt = min(32, cur.kk - base);
                    float2 tv = fc.wv;
                    if (base > 1) tv = lane < cnt ? Tc[cur.QB - base - lane] : make_float2(1.f, 0.f);
                    for (int l = 0; l < cnt; ++l)
                        C = carry_step(C, {__shfl_sync(0xffffffffu, tv.x, l), __shfl_sync(0xffffffffu, tv.y, l)});
                }
            }
            if (GATED && cur.kk >= 1 && lane == 0)
                a.ctab[((int64_t)cur.slot * nqt + cur.QB) * nqt + cur.QB - cur.kk] = make_float2(C.re, C.im);
            ok = produce_tile<DP, GATED, L>(a, maps, m, tmem, bh, cur.QB, cur.kk, C, k, kph, fc, rowdata,
                                            a.withhold_stats);
            if (GATED && cur.kk >= 1) C = carry_step(C, {fc.ct.x, fc.ct.y});
        }
    } else {
        const int q = warp & 3, h = warp >> 2;
        const int i = 32 * q + lane;  // local row
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16) + 64 * h;
        int k = 0, uc = 0;
        bool ok = true;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++uc) {
            const int slot = u / per_head;
            int QB, c;
            stats_unit(u - slot * per_head, nqt, CH, QB, c);
            const float scale2 = tab.qk[slot] * 1.4426950408889634f / sqrtf((float)a.d);
            const bool valid = QB * 128 + i < n;
            const int k0 = c * CH, k1 = min(c * CH + CH, QB + 1);
            float M = -INFINITY, Z = 0.f, chk = 0.f;
            for (int kk = k0; kk < k1; ++kk, ++k) {
                const int b = k & 1;
                if (ok) ok = wait_bar_warp(m.sfull + b, (k >> 1) & 1, m.abort, a.status, 0);
                if (!ok) continue;
                tc_fence_after();
                const int kind = m.kind[b];
                if (kind == kTileOff) {
                    // paired lanes: t = s scale2 and R = |prefix_i| |C suffix_j|. When every
                    // product R of the warp's rows is positive (rq * min_j |c_j| > 0: rounding
                    // is monotone) the live mask drops out and R_i = rq sum_j |c_j| 2^{t - M}
                    // takes rq out of the sum; otherwise dead entries get t = -inf.
                    const float rq = m.rq[b * 128 + i];
                    const bool all_live = GATED ? rq * m.cmin[b] > 0.f : rq > 0.f;
                    const bool fast = __all_sync(0xffffffffu, all_live);
                    const float2 sc2 = make_float2(scale2, scale2), rq2 = make_float2(rq, rq);
                    const float2 zero2 = make_float2(0.f, 0.f), one2 = make_float2(1.f, 1.f);
                    const float *cmb = m.colm + b * 128 + 64 * h;
                    float2 chk2 = zero2;
                    for (int cc = 0; cc < 2; ++cc) {
                        float sv[32];
                        tmem_ld32f(trow + b * 128 + 32 * cc, sv);
                        float2 tt[16], ww[16];
                        float cmax = -INFINITY;
#pragma unroll
                        for (int e = 0; e < 16; ++e) {
                            tt[e] = mul2(make_float2(sv[2 * e], sv[2 * e + 1]), sc2);
                            chk2 = fma2(tt[e], zero2, chk2);
                            ww[e] = GATED ? *reinterpret_cast<const float2 *>(cmb + 32 * cc + 2 * e) : one2;
                            if (!fast) {
                                const float2 rr = mul2(rq2, ww[e]);
                                tt[e].x = rr.x > 0.f ? tt[e].x : -INFINITY;
                                tt[e].y = rr.y > 0.f ? tt[e].y : -INFINITY;
                                ww[e] = rr;
                            }
                            cmax = max3f(cmax, tt[e].x, tt[e].y);
                        }
                        if (cmax > M) {
                            Z = (M == -INFINITY) ? 0.f : Z * ex2_approx(M - cmax);
                            M = cmax;
                        }
                        if (M != -INFINITY) {
                            const float2 nm = make_float2(-M, -M);
                            float2 z2 = zero2;
#pragma unroll
                            for (int e = 0; e < 16; ++e) {
                                const float2 dd = add2(tt[e], nm);
                                z2 = fma2(ww[e], make_float2(ex2_approx(dd.x), ex2_approx(dd.y)), z2);
                            }
                            Z = fmaf(fast ? rq : 1.f, z2.x + z2.y, Z);
                        }
                    }
                    chk += chk2.x + chk2.y;
                } else if (kind == kTileDiag && !(q < 2 && h == 1)) {
                    // R_ij from j = i down: the same steps whichever half holds column j
                    float R = 1.f;
                    if (GATED && h == 0)
                        for (int j = min(i - 1, 127); j >= 64; --j) R *= m.colm[b * 128 + j + 1];
                    for (int cc = 1; cc >= 0; --cc) {
                        float sv[32], tt[32], rr[32];
                        tmem_ld32f(trow + b * 128 + 32 * cc, sv);
#pragma unroll
                        for (int e = 31; e >= 0; --e) {
                            const int j = 64 * h + 32 * cc + e;
                            if (GATED && j < i) R *= m.colm[b * 128 + j + 1];
                            tt[e] = sv[e] * scale2;
                            const bool causal = valid && j <= i;
                            if (causal) chk = fmaf(tt[e], 0.f, chk);
                            rr[e] = causal ? R : 0.f;
                        }
                        absorb32(M, Z, tt, rr);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(m.sempty + b);
            }
            // the two column halves of each row meet; half 0 writes the unit's partial
            float4 *xc = m.xchg + (uc & 1) * 128;
            if (h == 1) xc[i] = make_float4(M, Z, chk, 0.f);
            named_bar_sync(1, kConsumers);
            if (h == 0 && ok) {
                const float4 o = xc[i];
                merge_stats(M, Z, o.x, o.y);
                if (isnan(chk + o.z)) M = __int_as_float(0x7fc00000);
                a.part[(((int64_t)slot * nqt + QB) * NCH + c) * 128 + i] = make_float2(M, Z);
            }
        }
    }
    op_teardown(m, tmem);
}

// ================================================================ row data

// Per row of each query tile: the partials merged into (M, Z'), then the log2 of the row
// factor, E = (1-beta) M - beta log2 Z' (M at beta = 0), and prefix_i for the write, and
// |prefix_i| for its live test. One thread per row. The write forms each entry as
// 2^{(t - M) + E} = 2^{t - beta log2 Z} in one exponential, so an entry is +-inf only where
// its own value overflows (a row factor that overflows on its own never meets an entry that
// underflows: no inf * 0).
template <bool GATED>
__global__ void __launch_bounds__(128)
operator_rows_kernel(OpArgs a, const __grid_constant__ HeadTable tab)
{
    const int n = a.n, nqt = (n + 127) / 128, NCH = (nqt + a.chunk - 1) / a.chunk;
    const int slot = blockIdx.x / nqt, QB = blockIdx.x - slot * nqt;
    const int r = threadIdx.x, row = QB * 128 + r;
    const bool valid = row < n;
    const int bh = tab.bh[slot];
    const float beta = tab.beta[slot];
    const int64_t base = (int64_t)slot * nqt + QB;
    const float2 *part = a.part + base * NCH * 128;
    const int nch = QB / a.chunk + 1;
    float2 pv[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) pv[c] = c < nch ? part[c * 128 + r] : make_float2(-INFINITY, 0.f);
    cplx pq = {valid ? 1.f : 0.f, 0.f};
    if (GATED && valid) {
        const float2 p = a.prefix[(int64_t)bh * n + row];
        pq = {p.x, p.y};
    }
    float M = -INFINITY, Z = 0.f;
#pragma unroll
    for (int c = 0; c < 8; ++c) merge_stats(M, Z, pv[c].x, pv[c].y);
    const float E = (beta == 0.f) ? M : (1.f - beta) * M - beta * log2f(Z);
    a.rowf[base * 128 + r] = make_float4(M, E, pq.re, pq.im);
    a.rowq[base * 128 + r] = GATED ? cabs(pq) : pq.re;
    if (valid && (!isfinite(M) || !(Z > 0.f) || !isfinite(Z))) flag_status(a.status, RS_STATUS_NONFINITE_BIT);
}

// ================================================================ write

template <int DP, bool GATED, bool TMA_OUT>
__global__ void __launch_bounds__(kOpThreads, 1)
operator_kernel(OpArgs a, const __grid_constant__ HeadTable tab, const __grid_constant__ OpMaps maps)
{
    using L = OpLayout<DP, false>;
    constexpr int NSLOT = L::nslot;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    const OpSmem m = op_smem<L>(smem_raw);
    const uint32_t tmem = op_setup<L, true>(m, maps);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int n = a.n, nqt = (n + 127) / 128;
    const int per_head = nqt * nqt;
    const int tiles = per_head * tab.count;

    if (warp == kProdWarp) {
        // the CTA's lower tiles (KB <= QB), each tile's global data fetched one tile ahead;
        // the consumers store the tiles above the diagonal by themselves
        auto next_lower = [&](int t) {
            for (; t < tiles; t += gridDim.x) {
                const int rem = t % per_head, QB = rem / nqt;
                if (rem - QB * nqt <= QB) return t;
            }
            return tiles;
        };
        auto fetch = [&](int t, TileFetch &f) {
            const int slot = t / per_head, rem = t - slot * per_head;
            const int QB = rem / nqt, kk = rem - QB * nqt;
            const int bh = tab.bh[slot];
            fetch_cols<GATED>(a, (int64_t)bh * n, QB, kk, f);
            const int64_t rbase = ((int64_t)slot * nqt + QB) * 128;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f.rf[e] = a.rowf[rbase + lane + 32 * e];
                f.rq[e] = a.rowq[rbase + lane + 32 * e];
            }
            f.ct = make_float2(1.f, 0.f);
            if (GATED && kk >= 1) f.ct = a.ctab[((int64_t)slot * nqt + QB) * nqt + QB - kk];
        };
        auto rowdata = [&](const TileFetch &f, int b) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                m.rows[b * 128 + lane + 32 * e] = f.rf[e];
                m.rq[b * 128 + lane + 32 * e] = f.rq[e];
            }
        };
        uint32_t kph = 0;
        bool ok = true;
        int t = next_lower(blockIdx.x);
        TileFetch fn;
        if (t < tiles) fetch(t, fn);
        for (int k = 0; ok && t < tiles; ++k) {
            const int tc = t;
            const TileFetch fc = fn;
            t = next_lower(t + gridDim.x);
            if (t < tiles) fetch(t, fn);
            const int slot = tc / per_head, rem = tc - slot * per_head;
            const int QB = rem / nqt, kk = rem - QB * nqt;
            ok = produce_tile<DP, GATED, L>(a, maps, m, tmem, tab.bh[slot], QB, kk, {fc.ct.x, fc.ct.y}, k,
                                            kph, fc, rowdata, a.withhold_write);
        }
    } else {
        const int q = warp & 3, h = warp >> 2;
        const int i = 32 * q + lane;  // local row
        const uint32_t trow = tmem + ((uint32_t)(32 * q) << 16) + 64 * h;
        const uint32_t zero = m.sbase + L::zero;
        const uint32_t stg0 = m.sbase + L::staging + (uint32_t)warp * NSLOT * 8192;
        int k = 0, nst = 0;
        bool ok = true;
        // a 32 x 32 block of zeros of both planes at column x0, row y0
        auto put_zero = [&](int x0, int y0, int bh) {
            if (TMA_OUT) {
                if (lane == 0) {
                    tma_store_3d(&maps.wre, zero, x0, y0, bh);
                    tma_store_3d(&maps.wim, zero, x0, y0, bh);
                    bulk_commit_group();
                }
            } else {
                const int col = x0 + lane;
                float *wr = a.W_re + (int64_t)bh * n * n, *wi = a.W_im + (int64_t)bh * n * n;
                if (col < n)
                    for (int r = 0; r < 32 && y0 + r < n; ++r) {
                        wr[(int64_t)(y0 + r) * n + col] = 0.f;
                        wi[(int64_t)(y0 + r) * n + col] = 0.f;
                    }
            }
        };
        // a 32 x 32 block at column x0, row y0: this lane gives its row (vr, and vi unless
        // im_zero) through a staging slot
        auto put = [&](int x0, int y0, int bh, const float (&vr)[32], const float (&vi)[32], bool im_zero) {
            const uint32_t slot = stg0 + (uint32_t)(nst % NSLOT) * 8192;
            ++nst;
            if (TMA_OUT) {
                if (lane == 0) bulk_wait_read<NSLOT - 1>();  // the slot's last store has read it
                __syncwarp();
            }
            const uint32_t rowa = slot + (uint32_t)lane * 128;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint32_t off = (uint32_t)((c ^ (lane & 7)) << 4);
                sts128(rowa + off, make_uint4(__float_as_uint(vr[4 * c]), __float_as_uint(vr[4 * c + 1]),
                                              __float_as_uint(vr[4 * c + 2]), __float_as_uint(vr[4 * c + 3])));
                if (!im_zero)
                    sts128(rowa + 4096 + off,
                           make_uint4(__float_as_uint(vi[4 * c]), __float_as_uint(vi[4 * c + 1]),
                                      __float_as_uint(vi[4 * c + 2]), __float_as_uint(vi[4 * c + 3])));
            }
            if (TMA_OUT) {
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&maps.wre, slot, x0, y0, bh);
                    tma_store_3d(&maps.wim, im_zero ? zero : slot + 4096, x0, y0, bh);
                    bulk_commit_group();
                }
            } else {
                __syncwarp();
                const int col = x0 + lane;
                float *wr = a.W_re + (int64_t)bh * n * n, *wi = a.W_im + (int64_t)bh * n * n;
                const float *sm = reinterpret_cast<const float *>(m.base + (slot - m.sbase));
                if (col < n)
                    for (int r = 0; r < 32 && y0 + r < n; ++r) {
                        const int e = r * 32 + (((lane >> 2) ^ (r & 7)) << 2) + (lane & 3);
                        wr[(int64_t)(y0 + r) * n + col] = sm[e];
                        wi[(int64_t)(y0 + r) * n + col] = im_zero ? 0.f : sm[1024 + e];
                    }
                __syncwarp();
            }
        };

        for (int t = blockIdx.x; ok && t < tiles; t += gridDim.x) {
            const int slot = t / per_head, rem = t - slot * per_head;
            const int QB = rem / nqt, kk = rem - QB * nqt;
            const int bh = tab.bh[slot];
            const int y0 = QB * 128 + 32 * q;
            if (kk > QB) {  // above the diagonal
                put_zero(kk * 128 + 64 * h, y0, bh);
                put_zero(kk * 128 + 64 * h + 32, y0, bh);
                continue;
            }
            const int KB = QB - kk, b = k & 1;
            ok = wait_bar_warp(m.sfull + b, (k >> 1) & 1, m.abort, a.status, 0);
            ++k;
            if (!ok) break;
            tc_fence_after();
            const int kind = m.kind[b];
            const int x0 = KB * 128 + 64 * h;
            if (kind == kTileZero || (kind == kTileDiag && q < 2 && h == 1)) {
                put_zero(x0, y0, bh);
                put_zero(x0 + 32, y0, bh);
            } else {
                const float scale2 = tab.qk[slot] * 1.4426950408889634f / sqrtf((float)a.d);
                const float4 rs = m.rows[b * 128 + i];  // M, E, prefix_i
                const float M = rs.x, E = rs.y;
                if (kind == kTileOff) {
                    const float rq = m.rq[b * 128 + i];
                    const bool fast = __all_sync(0xffffffffu, GATED ? rq * m.cmin[b] > 0.f : true);
                    const float2 fre = make_float2(rs.z, rs.z), fim = make_float2(rs.w, rs.w);
                    for (int cc = 0; cc < 2; ++cc) {
                        float sv[32], vr[32], vi[32];
                        tmem_ld32f(trow + b * 128 + 32 * cc, sv);
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int j = 64 * h + 32 * cc + e;
                            const float tl = fminf(fmaf(sv[e], scale2, -M), 0.f);
                            if (GATED) {
                                // W_ij = (prefix_i) (C suffix_j) 2^{t - M + E}, in paired lanes;
                                // a component of G that is exactly 0 stays 0 (no 0 * inf)
                                const float4 c = m.col[b * 128 + j];
                                const bool live = fast || rq * m.colm[b * 128 + j] > 0.f;
                                const float p = live ? ex2_approx(tl + E) : 0.f;
                                const float2 w = fma2(fre, make_float2(c.x, c.y), mul2(fim, make_float2(c.z, c.w)));
                                const float2 wp = mul2(w, make_float2(p, p));
                                vr[e] = w.x == 0.f ? 0.f : wp.x;
                                vi[e] = w.y == 0.f ? 0.f : wp.y;
                            } else {
                                vr[e] = ex2_approx(tl + E);
                                vi[e] = 0.f;
                            }
                        }
                        put(x0 + 32 * cc, y0, bh, vr, vi, !GATED);
                    }
                } else {
                    // the diagonal tile: G_ij one gate at a time from j = i down
                    cplx G = {1.f, 0.f};
                    float R = 1.f;
                    if (GATED && h == 0)
                        for (int j = min(i - 1, 127); j >= 64; --j) {
                            const float4 an = m.col[b * 128 + j + 1];
                            G = diag_step(G, {an.x, an.y});
                            R *= m.colm[b * 128 + j + 1];
                        }
                    for (int cc = 1; cc >= 0; --cc) {
                        float sv[32], vr[32], vi[32];
                        tmem_ld32f(trow + b * 128 + 32 * cc, sv);
#pragma unroll
                        for (int e = 31; e >= 0; --e) {
                            const int j = 64 * h + 32 * cc + e;
                            if (GATED && j < i) {
                                const float4 an = m.col[b * 128 + j + 1];
                                G = diag_step(G, {an.x, an.y});
                                R *= m.colm[b * 128 + j + 1];
                            }
                            const bool live = j <= i && R > 0.f;
                            const float p = live ? ex2_approx(fminf(fmaf(sv[e], scale2, -M), 0.f) + E) : 0.f;
                            vr[e] = GATED ? (G.re == 0.f ? 0.f : G.re * p) : p;
                            vi[e] = GATED ? (G.im == 0.f ? 0.f : G.im * p) : 0.f;
                        }
                        put(x0 + 32 * cc, y0, bh, vr, vi, !GATED);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(m.sempty + b);
        }
        if (TMA_OUT && lane == 0) bulk_wait_all();
        __syncwarp();
    }
    op_teardown(m, tmem);
}

template <int DP, bool GATED>
cudaError_t launch_stats(const OpArgs &a, const HeadTable &tab, const OpMaps &maps, cudaStream_t s)
{
    using L = OpLayout<DP, true>;
    auto k = operator_stats_kernel<DP, GATED>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::alloc);
    if (e != cudaSuccess) return e;
    const int nqt = (a.n + 127) / 128, NCH = (nqt + a.chunk - 1) / a.chunk;
    int per_head = 0;
    for (int c = 0; c < NCH; ++c) per_head += nqt - c * a.chunk;
    const int units = per_head * tab.count;
    const int grid = std::max(1, std::min(units, 2 * device_sm_count()));
    k<<<grid, kOpThreads, L::alloc, s>>>(a, tab, maps);
    return cudaGetLastError();
}

template <bool GATED>
cudaError_t launch_rows(const OpArgs &a, const HeadTable &tab, cudaStream_t s)
{
    const int nqt = (a.n + 127) / 128;
    operator_rows_kernel<GATED><<<nqt * tab.count, 128, 0, s>>>(a, tab);
    return cudaGetLastError();
}

template <int DP, bool GATED, bool TMA_OUT>
cudaError_t launch_write(const OpArgs &a, const HeadTable &tab, const OpMaps &maps, cudaStream_t s)
{
    using L = OpLayout<DP, false>;
    auto k = operator_kernel<DP, GATED, TMA_OUT>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::alloc);
    if (e != cudaSuccess) return e;
    const int nqt = (a.n + 127) / 128;
    const int64_t tiles = (int64_t)nqt * nqt * tab.count;
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(tiles, device_sm_count()));
    k<<<grid, kOpThreads, L::alloc, s>>>(a, tab, maps);
    return cudaGetLastError();
}

template <int DP, bool GATED>
cudaError_t launch_write_out(const OpArgs &a, const HeadTable &tab, const OpMaps &maps, cudaStream_t s)
{
    return a.tma_out ? launch_write<DP, GATED, true>(a, tab, maps, s)
                     : launch_write<DP, GATED, false>(a, tab, maps, s);
}

}  // namespace

int operator_chunk(int n)
{
    const int nqt = (n + 127) / 128;
    return std::max(4, (nqt + 7) / 8);
}

cudaError_t launch_operator_stats(const OpArgs &a, const HeadTable &tab, const OpMaps &maps, int dpad,
                                  cudaStream_t s)
{
    if (tab.count == 0 || a.n == 0) return cudaSuccess;
    const bool gated = tab.g[0] != 0.f;
    cudaError_t e;
    if (dpad == 64)
        e = gated ? launch_stats<64, true>(a, tab, maps, s) : launch_stats<64, false>(a, tab, maps, s);
    else
        e = gated ? launch_stats<128, true>(a, tab, maps, s) : launch_stats<128, false>(a, tab, maps, s);
    if (e != cudaSuccess) return e;
    return gated ? launch_rows<true>(a, tab, s) : launch_rows<false>(a, tab, s);
}

cudaError_t launch_operator(const OpArgs &a, const HeadTable &tab, const OpMaps &maps, int dpad,
                            cudaStream_t s)
{
    if (tab.count == 0 || a.n == 0) return cudaSuccess;
    const bool gated = tab.g[0] != 0.f;
    if (dpad == 64)
        return gated ? launch_write_out<64, true>(a, tab, maps, s) : launch_write_out<64, false>(a, tab, maps, s);
    return gated ? launch_write_out<128, true>(a, tab, maps, s) : launch_write_out<128, false>(a, tab, maps, s);
}

}  // namespace rs
