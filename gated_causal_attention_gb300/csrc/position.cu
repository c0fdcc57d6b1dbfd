// position.cu -- position-only heads as a causal convolution over a prefix normaliser (K5).
//
// "A position-only causal softmax head is a causal convolution divided by a prefix
// normalizer" (proofs.blah.dev, theorem pos-head-is-causal-convolution), with the switches
// of "Resolvent Operator" at g = 0: when the logit of query i and key j is qk * a(i - j),
//     O_i = sum_{j<=i} e^{qk a(i-j)} v_j / Z_i^beta,  Z_i = sum_{d<=i} e^{qk a(d)},
// i.e. a causal convolution of v with the kernel e^{qk a(d)}, over a prefix sum of the same
// kernel. Two launches per table of heads:
//   prep  -- one CTA per head: M = max_d qk a(d); kappa(d) = e^{qk a(d) - M} rounded to bf16
//            (the tensor-core operand); C(i) = sum_{d<=i} kappa(d) over the rounded values, so
//            that the weights of a row sum to exactly what divides them; and the last offset
//            whose kappa is not 0;
//   main  -- one CTA per pair of 128-row query tiles: O_tile = sum_delta P(delta) V(Q - delta),
//            P(delta) the 128 x 128 block-Toeplitz tile P[r][c] = kappa(128 delta + r - c) (0
//            for a negative offset or one past n). Builder warps write P into shared memory
//            from the bf16 kappa table (no logits, no exponential per entry); one thread issues
//            the products transposed, O^T += V^T P^T (tcgen05.mma, V by TMA), so that both tiles
//            of the pair share each V tile; blocks whose offsets all lie past the last nonzero
//            kappa are skipped. The epilogue divides by C(i)^beta, multiplies by e^{(1-beta) M},
//            and writes O with coalesced 16-byte stores.
//            P stays out of TMEM: stores into TMEM from threads are starved while the tensor
//            pipe runs, so a P block written there would wait for the pipe's gaps.
#include "head_common.cuh"

namespace rs {

namespace {

using namespace head;

constexpr int kPrepThreads = 1024;

// One head per CTA. kap_bf16, C: [slots][n]; meta: [slots] = (M, last nonzero offset as a
// float-coded int) -- written as float2 (M, bit pattern of the offset).
__global__ void __launch_bounds__(kPrepThreads)
position_prep_kernel(PosArgs a, const __grid_constant__ HeadTable tab)
{
    __shared__ float s_red[32];
    __shared__ int s_bad, s_dmax;
    __shared__ float s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int slot = blockIdx.x, n = a.n;
    const float qk = tab.qk[slot];
    const float *av = a.a + (int64_t)(tab.bh[slot] % a.H) * n;
    __nv_bfloat16 *kap = a.kap + (int64_t)slot * a.kstride;
    float *C = a.C + (int64_t)slot * n;
    if (tid == 0) {
        s_bad = 0;
        s_dmax = -1;
        s_carry = 0.f;
    }
    // the largest logit, and the refusal of a non-finite a(d) or qk a(d)
    float mx = -INFINITY;
    bool bad = false;
    for (int d = tid; d < n; d += kPrepThreads) {
        const float x = av[d];
        const float t = qk * x;
        bad |= !isfinite(x) || !isfinite(t);
        mx = fmaxf(mx, t);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (lane == 0) s_red[warp] = mx;
    if (__syncthreads_or(bad) && tid == 0) s_bad = 1;
    if (warp == 0) {
        float m = s_red[lane];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) s_red[0] = m;
    }
    __syncthreads();
    const float M = s_red[0];
    if (s_bad) {  // refused: the main launch then builds no tile beyond the first
        if (tid == 0) {
            flag_status(a.status, RS_STATUS_NONFINITE_BIT);
            a.meta[slot] = make_float2(0.f, __int_as_float(-1));
        }
        for (int d = tid; d < a.kstride; d += kPrepThreads) kap[d] = __float2bfloat16_rn(0.f);
        for (int d = tid; d < n; d += kPrepThreads) C[d] = 0.f;
        return;
    }
    for (int d = n + tid; d < a.kstride; d += kPrepThreads) kap[d] = __float2bfloat16_rn(0.f);  // zero tail
    // kappa rounded to bf16, its inclusive prefix sum, the last nonzero offset
    for (int base = 0; base < n; base += kPrepThreads) {
        const int d = base + tid;
        float k = 0.f;
        if (d < n) {
            const __nv_bfloat16 kb = __float2bfloat16_rn(expf(qk * av[d] - M));
            kap[d] = kb;
            k = __bfloat162float(kb);
            if (k > 0.f) atomicMax(&s_dmax, d);
        }
        // block-wide inclusive scan: within warps, then over the warp totals
        float x = k;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        __syncthreads();  // s_red is reused
        if (lane == 31) s_red[warp] = x;
        __syncthreads();
        if (warp == 0) {
            float w = s_red[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const float y = __shfl_up_sync(0xffffffffu, w, o);
                if (lane >= o) w += y;
            }
            s_red[lane] = w;
        }
        __syncthreads();
        const float carry = s_carry;
        const float incl = carry + (warp > 0 ? s_red[warp - 1] : 0.f) + x;
        if (d < n) C[d] = incl;
        __syncthreads();
        if (tid == kPrepThreads - 1) s_carry = incl;
    }
    __syncthreads();
    if (tid == 0) a.meta[slot] = make_float2(M, __int_as_float(s_dmax));
}

template <int DVP>
struct PosCfg {
    static constexpr uint32_t v_bytes = (DVP / 64) * kRegion;  // one V tile: 128 keys x DVP bf16
    static constexpr int NSV = 3;                              // V stages
    static constexpr int NPB = 4;                              // P blocks
    // P block b, keys [64 kr, 64 kr + 64) of its 128 rows: p_ring + kr * p_half + b * kRegion,
    // so the rows of consecutive blocks b, b + 1 follow one another in each key half
    static constexpr uint32_t p_half = NPB * kRegion;
    static constexpr uint32_t v_ring = 0;
    static constexpr uint32_t p_ring = v_ring + NSV * v_bytes;
    static constexpr uint32_t rowf = p_ring + 2 * p_half;      // float [2][128] row factors
    static constexpr uint32_t bars = rowf + 2 * 128 * 4;       // vfull, vempty, pfull, pfree, accfull, drain
    static constexpr int nbars = 2 * NSV + 2 * NPB + 2;
    static constexpr uint32_t misc = bars + nbars * 8;         // tmem slot, abort flag
    static constexpr uint32_t end = misc + 16;
    static constexpr uint32_t alloc = end + 1024;
    // the epilogue stages both output tiles (fp32, [query][dv]) over the V and P rings
    static_assert(2 * 128 * DVP * 4 <= rowf, "epilogue staging");
    static_assert(alloc <= 227 * 1024, "shared memory");
};

constexpr int kPosThreads = 384;  // warpgroup 0: TMA (warp 0) and MMA (warp 1); 1-2: P builders
constexpr int kBarBuild = 1;

// One CTA takes two query tiles of one head, Qlo = 2m and Qhi = 2m + 1 (Qhi absent at the end
// of an odd tile count), and computes their outputs transposed, O^T = V^T P^T, so that the
// tensor core reads V (the A operand) once for both tiles: accumulator lane = value
// column, TMEM column = query (the lower tile's 128, then the upper tile's).
// Step j loads V(Qhi - j); the upper tile takes it with P(j) and the lower one with P(j - 1).
// Both are blocks of one causal Toeplitz matrix (entry kappa(query - key)): the upper tile's
// rows of step j - 1 are the lower tile's rows of step j, so each P block is built once, and
// when P(j - 1) and P(j) sit in consecutive buffers one N = 256 MMA covers both tiles.
// Tile A (query tile Q_A, lag L_A: 0 for the upper tile, 1 for the lower one when the upper
// exists) takes part at step j when 0 <= j - L_A <= D_A with
// D_A = min(Q_A, the last block offset whose kernel is not all 0).
template <int DVP>
__global__ void __launch_bounds__(kPosThreads, 1)
position_head_kernel(PosArgs a, const __grid_constant__ HeadTable tab, const __grid_constant__ PosMaps maps)
{
    using L = PosCfg<DVP>;
    constexpr int NSV = L::NSV, NPB = L::NPB;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t *vfull = reinterpret_cast<uint64_t *>(smem + L::bars);
    uint64_t *vempty = vfull + NSV, *pfull = vfull + 2 * NSV, *pfree = pfull + NPB, *accfull = pfree + NPB;
    uint64_t *drain = accfull + 1;  // the MMA issuer's own wait for its work when it winds down
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L::misc);
    volatile int *s_abort = reinterpret_cast<volatile int *>(smem + L::misc) + 1;
    float *s_rowf = reinterpret_cast<float *>(smem + L::rowf);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
    const int n = a.n, nqt = (n + 127) / 128, npairs = (nqt + 1) / 2;
    // blocks run head group by head group (a group's V stays in L2 while its query tiles
    // stream it), longest pairs first within a group
    const int G = a.heads_per_group;
    const int grp = (int)blockIdx.x / (G * npairs);
    const int rem = (int)blockIdx.x - grp * G * npairs;
    const int gsz = min(G, tab.count - grp * G);
    const int m = npairs - 1 - rem / gsz;
    const int slot = grp * G + rem % gsz;
    const int bh = tab.bh[slot];
    const float2 meta = a.meta[slot];  // (M, last offset whose kappa is not 0)
    const int dmaxt = max((__float_as_int(meta.y) + 127) / 128, 0);  // last nonzero block offset
    const int Qlo = 2 * m;
    const bool has_hi = Qlo + 1 < nqt;
    const int Qhi = has_hi ? Qlo + 1 : Qlo;
    const int Dlo = min(Qlo, dmaxt), Dhi = has_hi ? min(Qhi, dmaxt) : -1;
    const int Llo = has_hi ? 1 : 0;
    const int S = max(Llo + Dlo, Dhi) + 1;  // steps
    const int Dmax = max(Dlo, Dhi);         // P(0 .. Dmax) are built

    if (warp == 0 && lane == 0) {
        for (int i = 0; i < L::nbars; ++i) mbar_init(vfull + i, 1);
        for (int i = 0; i < NPB; ++i) mbar_init(pfull + i, 8);  // one arrival per builder warp
        *s_abort = 0;
        fence_mbar_init();
        prefetch_tmap(&maps.v);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (wg == 0) {
        if (warp == 0 && lane == 0) {
            // ------------------------------------------------------------ TMA: V(Qhi - j)
            int issued = 0;
            for (int j = 0; j < S; ++j) {
                const int sv = j % NSV;
                if (j == 1 && (int)blockIdx.x == a.withhold) break;  // test knob (timeout path)
                if (j >= NSV && !wait_bar(vempty + sv, ((j / NSV) - 1) & 1, s_abort, a.status, 256)) break;
                unsigned char *stg = smem + L::v_ring + sv * L::v_bytes;
                mbar_arrive_expect_tx(vfull + sv, L::v_bytes);
                for (int rr = 0; rr < DVP / 64; ++rr)
                    tma_load_3d(stg + rr * kRegion, &maps.v, vfull + sv, rr * 64, (Qhi - j) * 128, bh);
                ++issued;
            }
            drain_loads(vfull, NSV, issued);
        } else if (warp == 1 && lane == 0) {
            // ------------------------------------------------------------ MMA: O^T += V^T P^T
            constexpr uint32_t idesc1 = idesc_bf16(128, 128, true, false);  // one tile
            constexpr uint32_t idesc2 = idesc_bf16(128, 256, true, false);  // both tiles
            // V^T: value columns contiguous (64 per 128-byte row, 16 KB to the next 64; for
            // DVP = 64 the upper half of M reads the next buffer and lands in unused lanes)
            const uint64_t da0 = sw128_desc(sbase + L::v_ring, kRegion, 1024);
            // P^T: keys contiguous, 128-byte swizzled rows; the K-step offset is added later
            const uint64_t dp0 = sw128_desc(sbase + L::p_ring, 16, 1024);
            auto dp = [&](int b, int ks) {
                return dp0 + (((uint32_t)(ks >> 2) * L::p_half + (uint32_t)b * kRegion + (uint32_t)(ks & 3) * 32) >> 4);
            };
            bool ok = true;
            for (int j = 0; j < S; ++j) {
                const int sv = j % NSV;
                const int dl = j - Llo;
                const bool lo = dl >= 0 && dl <= Dlo, hi = has_hi && j <= Dhi;
                // P(j) is new at this step (P(dl) of the lower tile was waited for at step dl)
                if (!wait_bar(vfull + sv, (j / NSV) & 1, s_abort, a.status, 32) ||
                    ((hi || (lo && Llo == 0)) && !wait_bar(pfull + j % NPB, (j / NPB) & 1, s_abort, a.status, 32))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint64_t da = da0 + (((uint32_t)sv * L::v_bytes) >> 4);
                const int blo = (dl >= 0 ? dl : 0) % NPB;
                if (lo && hi && dl >= 1 && blo + 1 < NPB) {
                    // P(j - 1), P(j) in consecutive buffers: 256 consecutive query rows
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) umma_bf16_ss(tmem, da + (ks * 2048 >> 4), dp(blo, ks), idesc2, 1u);
                } else {
                    if (lo) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            umma_bf16_ss(tmem, da + (ks * 2048 >> 4), dp(blo, ks), idesc1, (dl > 0 || ks > 0) ? 1u : 0u);
                    }
                    if (hi) {
#pragma unroll
                        for (int ks = 0; ks < 8; ++ks)
                            umma_bf16_ss(tmem + 128, da + (ks * 2048 >> 4), dp(j % NPB, ks), idesc1, (j > 0 || ks > 0) ? 1u : 0u);
                    }
                }
                umma_commit(vempty + sv);
                if (lo) umma_commit(pfree + blo);  // the last use of P(dl)
            }
            if (ok) umma_commit(accfull);
            drain_mma(drain);
        }
    } else {
        // ------------------------------------------------------------ P builders
        // Thread (h, r): row r of every P(delta), keys [64h, 64h + 64): one 128-byte swizzled
        // row of key half h. With the kernel table read as 32-bit words, K32[w] =
        // (kappa(2w), kappa(2w + 1)) (zero-padded past n), key c of row r in block delta is
        // kappa(128 delta + r - c). The 33 words a row needs are read through the read-only
        // cache (the eight builder warps share them), a block ahead.
        const int h = wg - 1, r = tid & 127, bt = tid - 128;  // bt: 0..255 over the builders
        const uint32_t *K32 = reinterpret_cast<const uint32_t *>(a.kap + (int64_t)slot * a.kstride);
        // key pair (c, c+1), c = 64h + 2p: low half kappa(x), high half kappa(x - 1) with
        // x = 128 delta + r - c; x - 1 = 128 delta - 128 + e0 for e0 = r - c + 127, whose parity
        // is that of r + 1 for every pair of the row
        const int e0top = r - 64 * h + 127;  // e0 of the first pair; each next pair is 2 lower
        const bool odd = e0top & 1;
        // words of block t: index 64 t - 64 + ((e0top + 1) >> 1) - k, k = 0 .. 32 (odd rows use
        // 33 words, even rows the first 32)
        uint32_t wnext[33];
        auto fetch = [&](int t, uint32_t (&w)[33]) {
            const int w0 = 64 * t - 64 + ((e0top + 1) >> 1);
#pragma unroll
            for (int k = 0; k < 33; ++k) {
                const int wi = w0 - k;
                w[k] = wi >= 0 ? __ldg(K32 + wi) : 0u;  // negative offsets: 0 (causal)
            }
        };
        fetch(0, wnext);
        const uint32_t prow = sbase + L::p_ring + h * L::p_half + r * 128;
        bool ok = true;
        for (int t = 0; t <= Dmax; ++t) {
            const int pb = t % NPB;
            uint32_t wv[33];
#pragma unroll
            for (int k = 0; k < 33; ++k) wv[k] = wnext[k];
            if (t < Dmax) fetch(t + 1, wnext);
            // buffer pb last held P(t - NPB): the MMAs that read it are done
            if (t >= NPB && !wait_bar_warp(pfree + pb, ((t / NPB) - 1) & 1, s_abort, a.status, 0)) {
                ok = false;
                break;
            }
            uint32_t pk[32];
            if (odd) {
                // e0 odd: high half of word k+1 (kappa(x - 1)) with low half of word k (kappa(x))
#pragma unroll
                for (int p = 0; p < 32; ++p) pk[p] = __byte_perm(wv[p], wv[p + 1], 0x7610);
            } else {
                // e0 even: word k holds (kappa(x - 1), kappa(x)); swap its halves
#pragma unroll
                for (int p = 0; p < 32; ++p) pk[p] = __byte_perm(wv[p], 0u, 0x1032);
            }
            const uint32_t dst = prow + pb * kRegion;
#pragma unroll
            for (int c = 0; c < 8; ++c)
                sts128(dst + ((c ^ (r & 7)) << 4), make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]));
            fence_proxy_async_smem();  // the tensor core reads P through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(pfull + pb);
        }

        // ------------------------------------------------------------ epilogue
        // O_i = e^{(1-beta) M} (sum_d kappa(d) v_{i-d}) / C(i)^beta; an exact 0 stays 0. The
        // factor is applied as two equal halves f = e^{E/2}, O = (acc f) f, so that an output
        // within fp32 is not lost to a factor that alone overflows or underflows.
        // Thread (h, r) works out the factor of row r of the lower (h = 0) or upper (h = 1) tile.
        {
            const int QA = h ? Qhi : Qlo;
            const int row = QA * 128 + r;
            float f = 0.f;
            bool bad = false;
            if ((h == 0 || has_hi) && row < n) {
                const float beta = tab.beta[slot], M = meta.x;
                const float Ci = a.C[(int64_t)slot * n + row];
                bad = !(Ci > 0.f);  // every kappa of the row underflowed
                const float E = (beta == 0.f) ? M : (1.f - beta) * M - beta * logf(Ci);
                f = expf(0.5f * E);
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(a.status, RS_STATUS_NONFINITE_BIT);
            s_rowf[h * 128 + r] = f;
        }
        bool done = ok && wait_bar_warp(accfull, 0, s_abort, a.status, 0);
        // every MMA is done: the rings are free for staging; also publishes the row factors
        done = named_bar_and(kBarBuild, 256, done && !*s_abort);
        // Warpgroup h moves tile h out of TMEM, times its row factors: lane d (value column) of
        // TMEM columns [128 h, 128 h + 128), into a [query][DVP] fp32 block, 32 queries at a time
        float *stage = reinterpret_cast<float *>(smem + L::v_ring);
        const int d = (warp & 3) * 32 + lane;
        if (done && (h == 0 || has_hi)) {
            tc_fence_after();
            const uint32_t tcol = tmem + ((uint32_t)((warp & 3) * 32) << 16) + 128 * h;
            float *st = stage + h * 128 * DVP;
            const float *rf = s_rowf + h * 128;
#pragma unroll 1
            for (int qc = 0; qc < 4; ++qc) {
                uint32_t acc[32];
                RS_TMEM_LD32(tcol + 32 * qc, acc);  // warp-wide
                tmem_ld_wait();
                if (d < DVP) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const float x = __uint_as_float(acc[e]);
                        st[(32 * qc + e) * DVP + d] = x == 0.f ? 0.f : (x * rf[32 * qc + e]) * rf[32 * qc + e];
                    }
                }
            }
        }
        done = named_bar_and(kBarBuild, 256, done);
        if (done) {
            // coalesced stores: warp wi of the eight copies rows wi, wi + 8, ..., 16 bytes a lane
            const int wi = bt >> 5;
#pragma unroll 1
            for (int tt = 0; tt < (has_hi ? 2 : 1); ++tt) {
                const int Qt = tt ? Qhi : Qlo;
                const int nrows = min(128, n - Qt * 128);
                float *o0 = a.O + ((int64_t)bh * n + Qt * 128) * a.dv;
                const float *st = stage + tt * 128 * DVP;
                if (a.vec_out) {
#pragma unroll 1
                    for (int q = wi; q < nrows; q += 8) {
#pragma unroll
                        for (int c = 4 * lane; c < DVP; c += 128)
                            if (c < a.dv)
                                *reinterpret_cast<float4 *>(o0 + (int64_t)q * a.dv + c) =
                                    *reinterpret_cast<const float4 *>(st + q * DVP + c);
                    }
                } else {  // rows of dv % 4 != 0 floats: one value per store
#pragma unroll 1
                    for (int q = wi; q < nrows; q += 8)
                        for (int c = lane; c < a.dv; c += 32) o0[(int64_t)q * a.dv + c] = st[q * DVP + c];
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

template <int DVP>
cudaError_t launch_pos(const PosArgs &a, const HeadTable &tab, const PosMaps &maps, cudaStream_t s)
{
    using L = PosCfg<DVP>;
    position_prep_kernel<<<tab.count, kPrepThreads, 0, s>>>(a, tab);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    auto k = position_head_kernel<DVP>;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::alloc);
    if (e != cudaSuccess) return e;
    const int npairs = ((a.n + 127) / 128 + 1) / 2;
    k<<<npairs * tab.count, kPosThreads, L::alloc, s>>>(a, tab, maps);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_position_head(const PosArgs &a, const HeadTable &tab, const PosMaps &maps, int dvpad,
                                 cudaStream_t s)
{
    if (tab.count == 0 || a.n == 0) return cudaSuccess;
    return dvpad == 64 ? launch_pos<64>(a, tab, maps, s) : launch_pos<128>(a, tab, maps, s);
}

}  // namespace rs
