// head_fwd.cu -- the fused causal tiled resolvent head (K2) on the sm_103a tensor cores.
//
// "Resolvent Operator", section "Object": W_ij = G_ij e^{qk s_ij} / Z_i^beta and
// O_i = sum_{j<=i} W_ij V_j, evaluated in the log domain of section "Evaluation and
// refusals": the maximum of qk s_ij over the live entries (R_ij > 0) shifts the sum Z.
//
// One CTA owns one 128-row query tile QB of one head. Key tiles run from KB = QB-1 down to
// 0 (the off-diagonal tiles), then the diagonal tile KB = QB. The CTA is warp-specialised
// and software-pipelined (warpgroup 0 is the producer, 1 and 2 the softmax halves, 3 the
// value preparation of gated heads):
//   producer warp 0   TMA: Q once, then K and V tiles (one K+V ring for gated heads, a K
//                     ring and a V ring for g = 0 heads);
//   producer warp 1   issues S(t) = Q K(t)^T into one of 2-3 TMEM S buffers;
//   producer warp 2   issues O += P(t) V'(t) with P read from TMEM (it overwrites S). Two
//                     issuers, because a tcgen05.mma is accepted only about as fast as the
//                     pipe retires the previous one;
//   softmax halves    two threads per query row, keys [0,64) and [64,128) of each tile:
//                     live-masked running maximum M (moved only when it grows by more than
//                     2^8, so the accumulator is rarely rescaled), P = 2^{t - M} packed to
//                     bf16 into TMEM, the shifted sum Z', the row factor prefix_i, the
//                     diagonal tile and the epilogue;
//   value preparation thread j = key row j: c_j = C * suffix_j, V'_j = c_j V_j as [Re | Im]
//                     bf16 halves for one MMA with N = 2 dv, and the carry C <- C * (block
//                     total) for the next key tile.
// Across blocks the path product factors as prefix_i * C * suffix_j (gate_products.cuh);
// C only ever gains factors, so the key tiles beyond the first exactly-zero C are exactly
// dead and are never loaded. Inside the diagonal tile G_ij is formed one gate at a time
// from the top of each half down (rows of the upper half start the lower half from
// A_i = a_64 ... a_i), and two MMAs accumulate Re(P G) V and Im(P G) V.
// Heads with g = 0 have G = 1: no gate products, no value preparation, a real accumulator.
// The number of live off-diagonal key tiles of each query tile comes from a small launch
// before (head_numkv_kernel), so the CTA starts its loads right after one barrier.
// The epilogue stages O in the freed K/V ring and writes it with coalesced 16-byte stores.
//
// Every wait is bounded: one that runs out raises RS_STATUS_TIMEOUT, tells the other roles
// to stop, and the CTA winds down with its TMEM freed.
#include "head_common.cuh"

namespace rs {

namespace {

using namespace head;

// Warpgroup roles: 0 the producer (warp 0 loads by TMA, warp 1 issues S, warp 2 issues
// P V), 1 and 2 softmax (each query row has one thread in each:
// keys 0-63 and 64-127 of every key tile), 3 value preparation (gated heads only).
// After the prologue the producer (and value-prep) warpgroups hand registers to the softmax
// warpgroups (setmaxnreg); the shares add up to exactly what the launch provides:
//   gated:   512 threads x 128 = 2 x 128 x 184 + 128 x 80 + 128 x 64
//   ungated: 384 threads x 168 >= 2 x 128 x 216 + 128 x 64
template <bool GATED>
struct Roles {
    static constexpr int threads = GATED ? 512 : 384;
    static constexpr int prod_wg = 0;
    static constexpr int sm_wg0 = 1;  // softmax: warpgroups 1 and 2
    static constexpr int vprep_wg = 3;
    static constexpr int launch_regs = GATED ? 128 : 168;
    static constexpr int softmax_regs = GATED ? 184 : 216;
    static constexpr int vprep_regs = 80;
    static constexpr int prod_regs = 64;
    static_assert(2 * 128 * softmax_regs + (GATED ? 128 * vprep_regs : 0) + 128 * prod_regs <=
                      threads * launch_regs,
                  "register shares exceed the launch");
};
// Named barriers: all softmax threads; the value-prep warps; and, per lane quarter q, the two
// softmax warps (one per half) that hold rows 32q..32q+31.
constexpr int kBarSoftmax = 1, kBarVprep = 2, kBarRows0 = 3;

// (acc_re + i acc_im) <- z * (acc_re + i acc_im) over columns [c0, c1) of a row whose Re
// block starts at trow and Im block at trow + dvp (32 columns at a time)
__device__ __forceinline__ void cscale_acc_cols(uint32_t trow, int dvp, int c0, int c1, cplx z)
{
#pragma unroll 1
    for (int cc = c0; cc < c1; cc += 32) {
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

// A tile of a tensor map into L2 only (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_l2_3d(const CUtensorMap *map, int x, int y, int z)
{
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];"
                 ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z)
                 : "memory");
}

template <int DP, int DVP, bool GATED>
struct Cfg {
    static constexpr uint32_t q_bytes = (DP / 64) * kRegion;
    static constexpr uint32_t k_bytes = (DP / 64) * kRegion;
    static constexpr uint32_t v_bytes = (DVP / 64) * kRegion;
    static constexpr uint32_t small_bytes = 8192;
    static constexpr uint32_t budget = 227 * 1024 - 1024 - small_bytes - q_bytes;
    // Gated: Re V' replaces V in place and Im V' takes a region of its own when four such
    // stages fit; otherwise (when K is at least as wide as V) Re V' goes where K was, once
    // S(t) is done, and Im V' replaces V.
    static constexpr bool alias = DP >= DVP && budget / (k_bytes + 2 * v_bytes) < 4;
    static constexpr uint32_t extra = (GATED && !alias) ? v_bytes : 0;
    static constexpr uint32_t stage_bytes = k_bytes + v_bytes + extra;
    static constexpr int NS = (budget / stage_bytes) >= 4 ? 4 : (int)(budget / stage_bytes);
    static constexpr uint32_t stages = q_bytes;                       // stage s at stages + s*stage_bytes
    // Heads with g = 0 keep K and V in separate rings instead: a K stage frees as soon as its
    // S is done and a V stage once its P V is done, so the K loads run further ahead.
    static constexpr bool split = !GATED;
    static constexpr int NSV = 2;
    static constexpr int NSK_fit = (int)((budget - NSV * v_bytes) / k_bytes);
    static constexpr int NSK = NSK_fit >= 4 ? 4 : NSK_fit;
    static constexpr uint32_t vring = q_bytes + NSK * k_bytes;        // V stage s at vring + s*v_bytes
    static constexpr uint32_t small = split ? vring + NSV * v_bytes : stages + NS * stage_bytes;
    static constexpr uint32_t rc = small;                             // float [NS][128] |c_j|
    static constexpr uint32_t ga = rc + NS * 128 * 4;                 // float2 [128] gates of the query block
    static constexpr uint32_t gm = ga + 128 * 8;                      // float [128] |a|
    static constexpr uint32_t alllive = gm + 128 * 4;                 // int [NS]
    static constexpr uint32_t hmax = (alllive + NS * 4 + 15) & ~15u;  // float [2][2][128] half-row maxima
    static constexpr uint32_t zpart = hmax + 4 * 128 * 4;             // float [128] second half's Z'
    static constexpr uint32_t upA = zpart + 128 * 4;                  // float2 [128] prod a_{64..i}
    static constexpr uint32_t upR = upA + 128 * 8;                    // float [128] prod |a_{64..i}|
    static constexpr uint32_t bars = upR + 128 * 4;                   // mbarriers
    // q; full, empty, vprep, rc (4 each); s_full, p_full, pv_done (3 each); vfull, vempty
    // (4 each); diag_ready; the two MMA issuers' drains
    static constexpr int nbars = 1 + 4 * 4 + 3 * 3 + 2 * 4 + 1 + 2;
    static constexpr uint32_t misc = bars + nbars * 8;                // ints: tmem, -, abort, -, diag_all_live[4]
    static constexpr uint32_t end = misc + 64;
    static constexpr uint32_t alloc = end + 1024;
    static constexpr uint32_t acc_cols = GATED ? 2 * DVP : DVP;
    static constexpr uint32_t s_col0 = acc_cols;                      // S buffers: 128 columns each
    // Three S buffers where TMEM allows: S(t) then never waits for P(t-2) V to finish
    static constexpr int NSB = acc_cols <= 128 ? 3 : 2;
    // Re V' / Im V' offsets inside a stage, and the N-atom stride of the V' operand
    static constexpr uint32_t vre = alias ? 0 : k_bytes;
    static constexpr uint32_t vim = alias ? k_bytes : k_bytes + v_bytes;
    static constexpr uint32_t lbo_cplx = alias ? (DVP == 64 ? k_bytes : kRegion) : kRegion;
    static_assert(split ? NSK >= 2 : NS >= 2, "shared memory too small for two stages");
    static_assert(end <= 227 * 1024 - 1024, "shared memory budget");
    static_assert(end - small <= small_bytes, "small region budget");
    // the epilogue stages O in the K/V ring: Re and Im (gated) or Re and one zero chunk
    static constexpr uint32_t ring_bytes = split ? NSK * k_bytes + NSV * v_bytes : NS * stage_bytes;
    static_assert((GATED ? 2 * (DVP / 32) : DVP / 32 + 1) * kRegion <= ring_bytes, "epilogue staging");
    static_assert(acc_cols + NSB * 128 <= 512, "TMEM budget");
};

struct Barriers {
    // full/empty: the K+V ring (gated heads) or the K ring (g = 0); vfull/vempty: the V ring
    uint64_t *q, *full, *empty, *vprep, *rc, *s_full, *p_full, *pv_done, *vfull, *vempty;
    uint64_t *diag_ready;  // the value-prep warps have written the query block's gate data
    uint64_t *drain_s, *drain_pv;  // each MMA issuer's own wait for its work when it winds down
};

template <int DP, int DVP, bool GATED>
__global__ void __launch_bounds__(Roles<GATED>::threads, 1)
head_fwd_kernel(HeadArgs a, const __grid_constant__ HeadTable tab,
                const __grid_constant__ HeadMaps maps)
{
    using L = Cfg<DP, DVP, GATED>;
    using RL = Roles<GATED>;
    constexpr int NS = L::NS;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    uint64_t *bar0 = reinterpret_cast<uint64_t *>(smem + L::bars);
    Barriers B{bar0,      bar0 + 1,  bar0 + 5,  bar0 + 9,  bar0 + 13, bar0 + 17,
               bar0 + 20, bar0 + 23, bar0 + 26, bar0 + 30, bar0 + 34, bar0 + 35, bar0 + 36};
    int *misc = reinterpret_cast<int *>(smem + L::misc);
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(misc);
    volatile int *s_abort = misc + 2;
    int *s_diaglive = misc + 4;  // [4] per value-prep warp: its gates all have modulus >= 1/2
    float *s_rc = reinterpret_cast<float *>(smem + L::rc);
    float2 *s_ga = reinterpret_cast<float2 *>(smem + L::ga);
    float *s_gm = reinterpret_cast<float *>(smem + L::gm);
    int *s_alllive = reinterpret_cast<int *>(smem + L::alllive);
    float *s_hmax = reinterpret_cast<float *>(smem + L::hmax);  // [2 tiles][2 halves][128 rows]
    float *s_zpart = reinterpret_cast<float *>(smem + L::zpart);
    float2 *s_upA = reinterpret_cast<float2 *>(smem + L::upA);
    float *s_upR = reinterpret_cast<float *>(smem + L::upR);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, wg = warp >> 2;
    const int kTmaWarp = RL::prod_wg * 4, kMmaWarp = RL::prod_wg * 4 + 1, kPvWarp = RL::prod_wg * 4 + 2;
    const int n = a.n;
    const int nqt = (n + 127) / 128;
    // Blocks run head group by head group (the K/V of a group stays in L2 while its query
    // tiles stream it), longest query tiles first within a group.
    const int G = a.heads_per_group;
    const int grp = (int)blockIdx.x / (G * nqt);
    const int rem = (int)blockIdx.x - grp * G * nqt;
    const int gsz = min(G, tab.count - grp * G);
    const int QB = nqt - 1 - rem / gsz;
    const int slot = grp * G + rem % gsz;
    const int bh = tab.bh[slot];
    const float beta = tab.beta[slot], qk = tab.qk[slot];
    const int sQ = QB * 128;
    const int64_t tok0 = (int64_t)bh * n;

    // ------------------------------------------------------------ prologue
    if (warp == kTmaWarp && lane == 0) {
        for (int i = 0; i < L::nbars; ++i) {
            const uint64_t *b = bar0 + i;
            uint32_t count = 1;                                       // TMA / tcgen05.commit
            if (b >= B.vprep && b < B.vprep + 8) count = 4;           // value-prep warps (vprep, rc)
            if (b >= B.p_full && b < B.p_full + 3) count = 8;         // softmax warps, both halves
            if (b == B.diag_ready) count = 4;                          // value-prep warps
            mbar_init(bar0 + i, count);
        }
        *s_abort = 0;
        fence_mbar_init();
        prefetch_tmap(&maps.q);
        prefetch_tmap(&maps.k);
        prefetch_tmap(&maps.v);
        // Q does not depend on anything the prologue works out: start it now
        mbar_arrive_expect_tx(B.q, L::q_bytes);
        for (int r = 0; r < DP / 64; ++r)
            tma_load_3d(smem + r * kRegion, &maps.q, B.q, r * 64, sQ, bh);
    }
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_slot, 512);
        tmem_relinquish();
    }
    // softmax threads (two per row: one per half of the key tile): the row factor prefix_i
    const bool softmax = wg == RL::sm_wg0 || wg == RL::sm_wg0 + 1;
    const int r = tid & 127;  // query row (softmax) or key row (value prep)
    const int row = sQ + r;
    const bool valid = softmax && row < n;
    // off-diagonal key tiles: up to the first exactly-zero carry (gated heads, counted by
    // head_numkv_kernel), every earlier tile otherwise
    const int numkv = GATED ? a.numkv[slot * nqt + QB] : QB;
    const int T = numkv + 1;  // tiles: numkv off-diagonal, then the diagonal
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // Registers move from the producer (and value-prep) warps to the softmax warps: each role
    // starts with its setmaxnreg; the shares add up to exactly what the CTA was launched with.
    if (wg == RL::prod_wg) {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RL::prod_regs));
    if (warp == kTmaWarp) {
        // ------------------------------------------------------------ TMA producer
        // The block that starts about when this one ends (one block per SM: block index plus
        // the SM count) finds its Q tile and first K and V tiles in L2: prefetched once this
        // block's own first tile is on its way.
        auto prefetch_next = [&]() {
            const int nb = (int)blockIdx.x + a.prefetch_ahead;
            if (a.prefetch_ahead <= 0 || nb >= (int)gridDim.x) return;
            const int ngrp = nb / (G * nqt);
            const int nrem = nb - ngrp * G * nqt;
            const int ngsz = min(G, tab.count - ngrp * G);
            const int nQB = nqt - 1 - nrem / ngsz;
            const int nslot = ngrp * G + nrem % ngsz;
            const int nbh = tab.bh[nslot];
            const int nkv = GATED ? a.numkv[nslot * nqt + nQB] : nQB;
            const int nkb = nkv > 0 ? nQB - 1 : nQB;
            for (int rr = 0; rr < DP / 64; ++rr) {
                tma_prefetch_l2_3d(&maps.q, rr * 64, nQB * 128, nbh);
                tma_prefetch_l2_3d(&maps.k, rr * 64, nkb * 128, nbh);
            }
            for (int rr = 0; rr < DVP / 64; ++rr) tma_prefetch_l2_3d(&maps.v, rr * 64, nkb * 128, nbh);
        };
        if (lane == 0 && L::split) {  // the K ring
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int st = t % L::NSK;
                if (t == 1 && (int)blockIdx.x == a.withhold) break;  // test knob (timeout path)
                if (t >= L::NSK && !wait_bar(B.empty + st, ((t / L::NSK) - 1) & 1, s_abort, a.status, 256)) break;
                const int kb = t < numkv ? QB - 1 - t : QB;
                unsigned char *stg = smem + L::stages + st * L::k_bytes;
                mbar_arrive_expect_tx(B.full + st, L::k_bytes);
                for (int rr = 0; rr < DP / 64; ++rr)
                    tma_load_3d(stg + rr * kRegion, &maps.k, B.full + st, rr * 64, kb * 128, bh);
                ++issued;
                if (t == 0) prefetch_next();
            }
            drain_loads(B.full, L::NSK, issued);
        } else if (lane == 0) {
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int st = t % NS;
                if (t == 1 && (int)blockIdx.x == a.withhold) break;  // test knob (timeout path)
                if (t >= NS && !wait_bar(B.empty + st, ((t / NS) - 1) & 1, s_abort, a.status, 256)) break;
                const int kb = t < numkv ? QB - 1 - t : QB;
                unsigned char *stg = smem + L::stages + st * L::stage_bytes;
                mbar_arrive_expect_tx(B.full + st, L::k_bytes + L::v_bytes);
                for (int rr = 0; rr < DP / 64; ++rr)
                    tma_load_3d(stg + rr * kRegion, &maps.k, B.full + st, rr * 64, kb * 128, bh);
                for (int rr = 0; rr < DVP / 64; ++rr)
                    tma_load_3d(stg + L::k_bytes + rr * kRegion, &maps.v, B.full + st, rr * 64, kb * 128, bh);
                ++issued;
                if (t == 0) prefetch_next();
            }
            drain_loads(B.full, NS, issued);
        }
        if (lane == 0) drain_loads(B.q, 1, 1);  // Q, loaded in the prologue
    } else if (L::split && warp == kTmaWarp + 3) {
        // ------------------------------------------------------------ TMA producer, V ring
        if (lane == 0) {
            int issued = 0;
            for (int t = 0; t < T; ++t) {
                const int sv = t % L::NSV;
                if (t == 1 && (int)blockIdx.x == a.withhold) break;  // test knob (timeout path)
                if (t >= L::NSV && !wait_bar(B.vempty + sv, ((t / L::NSV) - 1) & 1, s_abort, a.status, 256)) break;
                const int kb = t < numkv ? QB - 1 - t : QB;
                unsigned char *stg = smem + L::vring + sv * L::v_bytes;
                mbar_arrive_expect_tx(B.vfull + sv, L::v_bytes);
                for (int rr = 0; rr < DVP / 64; ++rr)
                    tma_load_3d(stg + rr * kRegion, &maps.v, B.vfull + sv, rr * 64, kb * 128, bh);
                ++issued;
            }
            drain_loads(B.vfull, L::NSV, issued);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer: S = Q K^T
        // A tcgen05.mma is accepted only about as fast as the tensor pipe retires the one
        // before it, so an issuing thread that stops to wait leaves the pipe idle. S and PV
        // therefore have a thread each: while one waits on its barriers the other issues.
        if (lane == 0) {
            constexpr uint32_t idesc_s = idesc_bf16(128, 128, false, false);
            // descriptors built once; a stage or K-step offset is added to the start-address
            // field (address >> 4 in bits 0-13, below 2^14 in shared memory)
            constexpr uint32_t kstride = L::split ? L::k_bytes : L::stage_bytes;  // K slot to K slot
            const uint64_t dq = sw128_desc(sbase, 16, 1024);
            const uint64_t dk0 = sw128_desc(sbase + L::stages, 16, 1024);
            const uint32_t tS = tmem + L::s_col0;
            constexpr int nsk = L::split ? L::NSK : NS;  // stages of the ring that holds K
            bool ok = wait_bar(B.q, 0, s_abort, a.status);
            for (int t = 0; ok && t < T; ++t) {
                const int st = t % nsk, sb = t % L::NSB;
                if (!wait_bar(B.full + st, (t / nsk) & 1, s_abort, a.status, 32)) break;
                // the S buffer last held P(t - NSB): its P V must be done
                if (t >= L::NSB && !wait_bar(B.pv_done + sb, ((t / L::NSB) - 1) & 1, s_abort, a.status, 32)) break;
                tc_fence_after();
                const uint64_t dk = dk0 + (((uint32_t)st * kstride) >> 4);
#pragma unroll
                for (int ks = 0; ks < DP / 16; ++ks) {
                    const uint32_t off = ((ks >> 2) * kRegion + (ks & 3) * 32) >> 4;
                    umma_bf16_ss(tS + sb * 128, dq + off, dk + off, idesc_s, ks > 0 ? 1u : 0u);
                }
                umma_commit(B.s_full + sb);
                if (L::split) umma_commit(B.empty + st);  // the K stage is free once S is done
            }
            drain_mma(B.drain_s);
        }
    } else if (warp == kPvWarp) {
        // ------------------------------------------------------------ MMA issuer: O += P V'
        if (lane == 0) {
            constexpr uint32_t idesc_pv = idesc_bf16(128, GATED ? 2 * DVP : DVP, false, true);
            constexpr uint32_t idesc_pv_half = idesc_bf16(128, DVP, false, true);
            constexpr uint32_t vstride = L::split ? L::v_bytes : L::stage_bytes;  // V slot to V slot
            const uint64_t dvraw0 = sw128_desc(sbase + (L::split ? L::vring : L::stages + L::k_bytes), kRegion, 1024);
            const uint64_t dvc0 = sw128_desc(sbase + L::stages + L::vre, L::lbo_cplx, 1024);
            const uint32_t tS = tmem + L::s_col0;
            for (int t = 0; t < T; ++t) {
                const int st = t % NS, sb = t % L::NSB, sv = t % L::NSV;
                if (!wait_bar(B.p_full + sb, (t / L::NSB) & 1, s_abort, a.status, 32)) break;
                if (GATED && t < numkv && !wait_bar(B.vprep + st, (t / NS) & 1, s_abort, a.status, 32)) break;
                if (L::split && !wait_bar(B.vfull + sv, (t / L::NSV) & 1, s_abort, a.status, 32)) break;
                tc_fence_after();
                const uint32_t vslot = (uint32_t)(L::split ? sv : st);
                const uint32_t acc0 = t > 0 ? 1u : 0u;
                const uint32_t pcol = tS + sb * 128;  // P overwrites its own S buffer
                if (t < numkv) {
                    const uint64_t dv = (GATED ? dvc0 : dvraw0) + ((vslot * vstride) >> 4);
                    umma_bf16_ts(tmem, pcol, dv, idesc_pv, acc0);
#pragma unroll
                    for (int ks = 1; ks < 8; ++ks)
                        umma_bf16_ts(tmem, pcol + ks * 8, dv + (ks * 2048 >> 4), idesc_pv, 1u);
                } else {  // diagonal tile: raw V, Re(P G) and Im(P G) from the two halves of P
                    const uint64_t dv = dvraw0 + ((vslot * vstride) >> 4);
                    umma_bf16_ts(tmem, pcol, dv, idesc_pv_half, acc0);
                    if (GATED) umma_bf16_ts(tmem + DVP, pcol + 64, dv, idesc_pv_half, acc0);
#pragma unroll
                    for (int ks = 1; ks < 8; ++ks) {
                        umma_bf16_ts(tmem, pcol + ks * 8, dv + (ks * 2048 >> 4), idesc_pv_half, 1u);
                        if (GATED)
                            umma_bf16_ts(tmem + DVP, pcol + 64 + ks * 8, dv + (ks * 2048 >> 4), idesc_pv_half, 1u);
                    }
                }
                umma_commit(B.pv_done + sb);
                umma_commit(L::split ? B.vempty + sv : B.empty + st);
            }
            drain_mma(B.drain_pv);
        }
    }
    } else if (GATED && wg == RL::vprep_wg) {
        // ------------------------------------------------------------ value preparation
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(RL::vprep_regs));
        const int j = r;
        cplx C = {1.f, 0.f};
        const float2 *Tc = a.carry + (int64_t)bh * nqt;
        // the suffix product of key j and the block total of the next key tile are loaded one
        // tile ahead, so their latency hides behind the current tile's work
        float2 sg_next = make_float2(0.f, 0.f), T_next = make_float2(0.f, 0.f);
        if (numkv > 0) {
            sg_next = a.suffix[tok0 + (QB - 1) * 128 + j];
            T_next = Tc[QB - 1];
        }
        for (int t = 0; t < numkv; ++t) {
            const int st = t % NS;
            const float2 sgv = sg_next, Tv = T_next;
            if (t + 1 < numkv) {
                sg_next = a.suffix[tok0 + (QB - 2 - t) * 128 + j];
                T_next = Tc[QB - 2 - t];
            }
            // a wait that runs out sets the abort flag; the group leaves together after the
            // barrier below, so no thread is left waiting on it. (The stage being full also
            // means the softmax rows are done with this stage's previous |c_j|.)
            wait_bar(B.full + st, (t / NS) & 1, s_abort, a.status, 128);
            const cplx c = key_scale(C, {sgv.x, sgv.y});
            const float rc = cabs(c);
            s_rc[st * 128 + j] = rc;
            const bool all = named_bar_and(kBarVprep, 128, rc > 0.f);
            if (*s_abort) break;
            s_alllive[st] = all;
            // the softmax rows need only |c_j|; the barrier above ordered every warp's writes
            if (lane == 0) mbar_arrive(B.rc + st);
            if (L::alias) wait_bar(B.s_full + t % L::NSB, (t / L::NSB) & 1, s_abort, a.status, 64);
            // V'_j = c_j V_j: Re and Im halves, same swizzled position as V_j; c_j rounded to
            // bf16 once, each product rounded to bf16
            const uint32_t stg = sbase + L::stages + st * L::stage_bytes;
            const uint32_t cre2 = pack_bf16x2(c.re, c.re), cim2 = pack_bf16x2(c.im, c.im);
#pragma unroll
            for (int rr = 0; rr < DVP / 64; ++rr) {
#pragma unroll
                for (int ch = 0; ch < 8; ++ch) {
                    // rows are 128 B apart: rotate the chunk order by the row so that a
                    // warp's 16-byte accesses spread over all banks
                    const uint32_t off = rr * kRegion + j * 128 + ((ch + j) & 7) * 16;
                    const uint4 v = lds128(stg + L::k_bytes + off);
                    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                    uint32_t ore[4], oim[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {  // two keys' elements per bf16x2 multiply
                        ore[e] = mul_bf16x2(w[e], cre2);
                        oim[e] = mul_bf16x2(w[e], cim2);
                    }
                    sts128(stg + L::vre + off, make_uint4(ore[0], ore[1], ore[2], ore[3]));
                    sts128(stg + L::vim + off, make_uint4(oim[0], oim[1], oim[2], oim[3]));
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.vprep + st);
            C = carry_step(C, {Tv.x, Tv.y});
        }
        // the query block's own gates, for the diagonal tile (read by the softmax rows once
        // diag_ready completes)
        {
            float2 av = make_float2(0.f, 0.f);
            if (sQ + r < n) av = a.gate[tok0 + sQ + r];
            s_ga[r] = av;
            const float am = cabs({av.x, av.y});
            s_gm[r] = am;
            // with every |a_k| >= 1/2, a product of at most 127 of them is at least 2^-127 > 0:
            // no diagonal-block entry j <= i is dead, and the softmax rows skip the live test
            // (one flag per value-prep warp)
            const bool big = __all_sync(0xffffffffu, am >= 0.5f || sQ + r >= n);
            if (lane == 0) s_diaglive[warp & 3] = big;
            if (r < 32) {
                // rows of the upper half of the block: A_i = a_64 a_65 ... a_i (and its modulus
                // product), so that keys of the lower half factor as A_i * prod_{k=j+1..63} a_k.
                // Lane l holds rows 64 + 2l and 65 + 2l; a warp scan over the pair products.
                const int i0 = 64 + 2 * r;
                float2 g0 = make_float2(0.f, 0.f), g1 = make_float2(0.f, 0.f);
                if (sQ + i0 < n) g0 = a.gate[tok0 + sQ + i0];
                if (sQ + i0 + 1 < n) g1 = a.gate[tok0 + sQ + i0 + 1];
                const cplx c0 = {g0.x, g0.y}, c1 = {g1.x, g1.y};
                const float m0 = cabs(c0), m1 = cabs(c1);
                cplx incl = cmul(c0, c1);
                float rincl = m0 * m1;
#pragma unroll
                for (int d = 1; d < 32; d <<= 1) {
                    const cplx y = shfl_up(incl, d);
                    const float ry = __shfl_up_sync(0xffffffffu, rincl, d);
                    if (r >= d) {
                        incl = cmul(y, incl);
                        rincl = ry * rincl;
                    }
                }
                cplx excl = shfl_up(incl, 1);
                float rexcl = __shfl_up_sync(0xffffffffu, rincl, 1);
                if (r == 0) {
                    excl = {1.f, 0.f};
                    rexcl = 1.f;
                }
                const cplx A0 = cmul(excl, c0);
                s_upA[i0] = make_float2(A0.re, A0.im);
                s_upA[i0 + 1] = make_float2(incl.re, incl.im);
                s_upR[i0] = rexcl * m0;
                s_upR[i0 + 1] = rincl;
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(B.diag_ready);
        }
    } else if (softmax) {
        // ------------------------------------------------------------ softmax rows
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(RL::softmax_regs));
        // the row factor prefix_i (loaded after the CTA's barrier: it is first needed with the
        // first tile's logits)
        cplx pq = {0.f, 0.f};
        float rq = 0.f;
        if (valid) {
            if (GATED) {
                const float2 v = a.prefix[tok0 + row];
                pq = {v.x, v.y};
                rq = cabs(pq);
            } else {
                pq = {1.f, 0.f};
                rq = 1.f;
            }
        }
        // Two threads per query row: half h takes keys [64h, 64h + 64) of every key tile.
        const int h = wg - RL::sm_wg0;
        const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
        const float scale2 = qk * 1.4426950408889634f / sqrtf((float)a.d);  // qk log2(e)/sqrt(d)
        // heads with qk = 0 never come here: they run as chains (O(n) readout)
        float M2 = -INFINITY;  // (stale) running live maximum, log2 units (same in both halves)
        float Zs = 0.f;        // this half's sum of R 2^{t - M}
        float chk = 0.f;       // turns NaN if an evaluated logit is not finite
        bool ok = true;

        for (int t = 0; t < numkv; ++t) {
            const int st = t % NS, sb = t % L::NSB;
            const uint32_t scol = trow + L::s_col0 + sb * 128;
            bool ready = wait_bar_warp(B.s_full + sb, (t / L::NSB) & 1, s_abort, a.status);
            if (GATED && ready) ready = wait_bar_warp(B.rc + st, (t / NS) & 1, s_abort, a.status);
            tc_fence_after();
            const float *rcs = s_rc + st * 128 + 64 * h;
            // fast: every entry of every valid row of this warp is live (no masking needed)
            const bool fast = !GATED || __all_sync(0xffffffffu, !ready || (s_alllive[st] && (rq > 0.f || !valid)));
            // this half's 64 logits stay in registers for both passes
            uint32_t s[64];
            if (ready) {
                RS_TMEM_LD32(scol + 64 * h, s);
                RS_TMEM_LD32(scol + 64 * h + 32, (s + 32));
                tmem_ld_wait();
            }
            // gated heads with dead entries (c_j = 0, or a row whose prefix is 0): their logits
            // are checked, then replaced by a value whose scaled logit is about -1e30, so that
            // they neither move the maximum nor give a P above 0. (Their P V and Z' terms carry
            // the factor c_j or prefix_i, which is 0, whatever P is.)
            bool any_live = true;
            if (GATED && !fast) {
                const float dead = fminf(fmaxf(-1e30f / scale2, -3e38f), 3e38f);
                const uint32_t wa = smem_u32(rcs);
                float cpd = 0.f;
                any_live = false;
#pragma unroll
                for (int e0 = 0; e0 < 64; e0 += 4) {
                    const uint4 wq = lds128(wa + e0 * 4);
                    const float w[4] = {__uint_as_float(wq.x), __uint_as_float(wq.y),
                                        __uint_as_float(wq.z), __uint_as_float(wq.w)};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const bool live = rq * w[k] > 0.f;
                        any_live |= live;
                        if (!live) {
                            cpd = fmaf(__uint_as_float(s[e0 + k]) * scale2, 0.f, cpd);
                            s[e0 + k] = __float_as_uint(dead);
                        }
                    }
                }
                chk += cpd;
            }
            // pass 1: the half-row live maximum of t = qk s log2(e): max (or min, for qk < 0)
            // of the raw logits, then one scaling; three-input extrema in four independent
            // chains keep the dependency chains short
            float mt;
            {
                float hx[4];
                if (scale2 >= 0.f) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) hx[e] = -INFINITY;
#pragma unroll
                    for (int e = 0; e < 64; e += 2)
                        hx[(e >> 1) & 3] = max3f(hx[(e >> 1) & 3], __uint_as_float(s[e]), __uint_as_float(s[e + 1]));
                    mt = max3f(hx[0], hx[1], fmaxf(hx[2], hx[3])) * scale2;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) hx[e] = INFINITY;
#pragma unroll
                    for (int e = 0; e < 64; e += 2)
                        hx[(e >> 1) & 3] = min3f(hx[(e >> 1) & 3], __uint_as_float(s[e]), __uint_as_float(s[e + 1]));
                    mt = min3f(hx[0], hx[1], fminf(hx[2], hx[3])) * scale2;
                }
            }
            if (!valid || !any_live) mt = -INFINITY;
            // the two halves exchange their maxima; the barrier also makes every S read of
            // this tile happen before either half writes P over it, and lets both halves
            // leave together if a wait ran out
            s_hmax[((t & 1) * 2 + h) * 128 + r] = mt;
            ok = named_bar_and(kBarRows0 + (warp & 3), 64, ready && !*s_abort);
            if (!ok) break;
            mt = fmaxf(mt, s_hmax[((t & 1) * 2 + (h ^ 1)) * 128 + r]);
            // move the maximum only when it grows by more than 2^8 (or is first set)
            float alpha = 1.f;
            if (mt > M2 + kRescaleLog2 || (M2 == -INFINITY && mt > -INFINITY)) {
                alpha = (M2 == -INFINITY) ? 0.f : ex2_approx(M2 - mt);
                M2 = mt;
                Zs *= alpha;
            }
            if (h == 0 && __any_sync(0xffffffffu, t > 0 && alpha != 1.f)) {
                // the accumulator holds P(<= t-1) V: wait for PV(t-1), then rescale
                if (wait_bar_warp(B.pv_done + (t - 1) % L::NSB, ((t - 1) / L::NSB) & 1, s_abort, a.status)) {
                    tc_fence_after();
                    scale_acc_row(trow, L::acc_cols, t > 0 ? alpha : 1.f);
                }
            }
            // pass 2: P = 2^{t - M} (bf16, two per TMEM column), Z' += |c_j| P.
            // A row with no live entry yet keeps M = -inf; its logits are still checked.
            // Rows past n take -inf as their shift, so that their P is 0 without a select.
            const float nMx = !valid ? -INFINITY : (M2 == -INFINITY) ? 0.f : -M2;
            const float2 sc2 = make_float2(scale2, scale2), nm2 = make_float2(nMx, nMx);
            const float2 z2 = make_float2(0.f, 0.f);
            float2 zp[2] = {z2, z2}, cp[2] = {z2, z2};  // partial sums, two lanes each
            uint32_t pk[32];
            // paired fp32 instructions: the logit scaling, the finiteness check and the Z'
            // sum each take one instruction per two keys
            auto pair = [&](int e, float2 w2) {
                const int k = (e >> 1) & 1;
                const float2 x2 = fma2(make_float2(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), sc2, nm2);
                cp[k] = fma2(x2, z2, cp[k]);
                const float2 p2 = make_float2(ex2_approx(x2.x), ex2_approx(x2.y));
                zp[k] = GATED ? fma2(w2, p2, zp[k]) : add2(zp[k], p2);
                pk[e >> 1] = pack_bf16x2(p2.x, p2.y);
            };
            if (!GATED) {
#pragma unroll
                for (int e = 0; e < 64; e += 4) {
                    pair(e, make_float2(1.f, 1.f));
                    pair(e + 2, make_float2(1.f, 1.f));
                }
            } else {
                // |c_j| of this half: shared loads issued 32 keys ahead of their use
                const uint32_t wa = smem_u32(rcs);
#pragma unroll
                for (int e0 = 0; e0 < 64; e0 += 32) {
                    uint4 wq[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) wq[q] = lds128(wa + (e0 + 4 * q) * 4);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        pair(e0 + 4 * q, make_float2(__uint_as_float(wq[q].x), __uint_as_float(wq[q].y)));
                        pair(e0 + 4 * q + 2, make_float2(__uint_as_float(wq[q].z), __uint_as_float(wq[q].w)));
                    }
                }
            }
            RS_TMEM_ST16(scol + 32 * h, pk);
            RS_TMEM_ST16(scol + 32 * h + 16, (pk + 16));
            Zs += (zp[0].x + zp[0].y) + (zp[1].x + zp[1].y);
            chk += (cp[0].x + cp[0].y) + (cp[1].x + cp[1].y);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(B.p_full + sb);  // one arrival per warp
        }

        // ------------------------------------------------ diagonal tile (both halves)
        // Half h takes keys [64h, 64h + 64) again; its 64 logits stay in registers for both
        // passes, so P is written over S in place once both halves have read theirs. G_ij is
        // formed one gate at a time from the top of the half down; a row of the upper half
        // starts the lower half's chain from A_i = prod_{k=64..i} a_k. The accumulator's row
        // factor is applied after pass 2, while the last off-diagonal P V drains.
        {
            const int t = numkv, sb = t % L::NSB;
            const uint32_t scol = trow + L::s_col0 + sb * 128;
            const int i = r, jtop = 64 * h + 63;
            const int jstop = i < jtop ? i : jtop;  // a_{j+1} enters the product for j < jstop
            const bool from_upper = GATED && h == 0 && i > 63;
            bool ready = ok && wait_bar_warp(B.s_full + sb, (t / L::NSB) & 1, s_abort, a.status);
            if (GATED && ready) ready = wait_bar_warp(B.diag_ready, 0, s_abort, a.status);
            tc_fence_after();
            uint32_t s[64];
            if (ready) {
                RS_TMEM_LD32(scol + 64 * h, s);
                RS_TMEM_LD32(scol + 64 * h + 32, (s + 32));
                tmem_ld_wait();
            }
            // pass 1: live maximum over j <= i
            const bool all_live = !GATED || (s_diaglive[0] && s_diaglive[1] && s_diaglive[2] && s_diaglive[3]);
            float mt = -INFINITY;
            if (ready && all_live) {
                // every entry j <= i is live: a causal extremum of the raw logits (max, or min
                // for qk < 0), scaled once
                float hx[4];
                if (scale2 >= 0.f) {
#pragma unroll
                    for (int e = 0; e < 4; ++e) hx[e] = -INFINITY;
#pragma unroll
                    for (int e = 0; e < 64; e += 2) {
                        const int j = 64 * h + e;
                        const float v0 = j <= i ? __uint_as_float(s[e]) : -INFINITY;
                        const float v1 = j + 1 <= i ? __uint_as_float(s[e + 1]) : -INFINITY;
                        hx[(e >> 1) & 3] = max3f(hx[(e >> 1) & 3], v0, v1);
                    }
                    mt = max3f(hx[0], hx[1], fmaxf(hx[2], hx[3])) * scale2;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e) hx[e] = INFINITY;
#pragma unroll
                    for (int e = 0; e < 64; e += 2) {
                        const int j = 64 * h + e;
                        const float v0 = j <= i ? __uint_as_float(s[e]) : INFINITY;
                        const float v1 = j + 1 <= i ? __uint_as_float(s[e + 1]) : INFINITY;
                        hx[(e >> 1) & 3] = min3f(hx[(e >> 1) & 3], v0, v1);
                    }
                    mt = min3f(hx[0], hx[1], fminf(hx[2], hx[3])) * scale2;
                }
                if (!valid || i < 64 * h) mt = -INFINITY;
            } else if (ready) {
                float R = from_upper ? s_upR[i] : 1.f;
#pragma unroll
                for (int e = 63; e >= 0; --e) {
                    const int j = 64 * h + e;
                    // branch-free steps (the factor loads do not wait on the chain)
                    if (GATED) {
                        const float Rn = R * s_gm[min(j + 1, 127)];
                        R = j < jstop ? Rn : R;
                    }
                    const bool live = valid && j <= i && R > 0.f;
                    mt = live ? fmaxf(mt, __uint_as_float(s[e]) * scale2) : mt;
                }
            }
            // the exchange also orders every S read of this tile before either half's P
            s_hmax[((t & 1) * 2 + h) * 128 + r] = mt;
            ok = named_bar_and(kBarRows0 + (warp & 3), 64, ready && !*s_abort);
            float alpha = 1.f;
            if (ok) {
                mt = fmaxf(mt, s_hmax[((t & 1) * 2 + (h ^ 1)) * 128 + r]);
                if (mt > M2 + kRescaleLog2 || (M2 == -INFINITY && mt > -INFINITY)) {
                    alpha = (M2 == -INFINITY) ? 0.f : ex2_approx(M2 - mt);
                    M2 = mt;
                    Zs *= alpha;
                }
                // the off-diagonal sums take the row factor |prefix_i| now; the diagonal
                // entries below carry their own R
                if (GATED) Zs *= rq;
                // pass 2: P = G 2^{t - M} on live entries: Re over columns [32h, 32h+32),
                // Im (gated) over [64 + 32h, 64 + 32h + 32)
                cplx G = from_upper ? cplx{s_upA[i].x, s_upA[i].y} : cplx{1.f, 0.f};
                float R = from_upper ? s_upR[i] : 1.f;
#pragma unroll
                for (int c = 1; c >= 0; --c) {
                    uint32_t pre[16], pim[16];
                    float odd_re = 0.f, odd_im = 0.f;  // key j+1 of the pair (j, j+1)
#pragma unroll
                    for (int e = 31; e >= 0; --e) {
                        const int j = 64 * h + 32 * c + e;
                        if (GATED) {
                            const float2 an = s_ga[min(j + 1, 127)];
                            const cplx Gn = diag_step(G, {an.x, an.y});
                            const float Rn = R * s_gm[min(j + 1, 127)];
                            G = j < jstop ? Gn : G;
                            R = j < jstop ? Rn : R;
                        }
                        const bool causal = valid && j <= i;
                        const float x = fmaf(__uint_as_float(s[32 * c + e]), scale2, -M2);
                        if (causal) chk = fmaf(x, 0.f, chk);
                        const bool live = causal && (all_live || R > 0.f);
                        const float p = live ? ex2_approx(x) : 0.f;
                        Zs = GATED ? fmaf(R, p, Zs) : Zs + p;
                        const float pr = GATED ? G.re * p : p;
                        const float pi = GATED ? G.im * p : 0.f;
                        // pack (j, j+1): the pair completes at even j
                        if (e & 1) {
                            odd_re = pr;
                            odd_im = pi;
                        } else {
                            pre[e >> 1] = pack_bf16x2(pr, odd_re);
                            pim[e >> 1] = pack_bf16x2(pi, odd_im);
                        }
                    }
                    RS_TMEM_ST16(scol + 32 * h + 16 * c, pre);
                    if (GATED) RS_TMEM_ST16(scol + 64 + 32 * h + 16 * c, pim);
                }
                tmem_st_wait();
                // the accumulator holds every off-diagonal P V: it takes alpha and (gated) the
                // row factor prefix_i, once the last of them is done
                // (gated: each half takes half of the columns)
                if ((GATED || h == 0) && numkv > 0 && (GATED || __any_sync(0xffffffffu, alpha != 1.f))) {
                    if (wait_bar_warp(B.pv_done + (t - 1) % L::NSB, ((t - 1) / L::NSB) & 1, s_abort, a.status)) {
                        tc_fence_after();
                        if (GATED)
                            cscale_acc_cols(trow, DVP, h * (DVP / 2), (h + 1) * (DVP / 2), cmul(pq, {alpha, 0.f}));
                        else
                            scale_acc_row(trow, L::acc_cols, alpha);
                    } else {
                        ok = false;
                    }
                }
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(B.p_full + sb);
        }

        // the second half hands its partial sum to the first, which works out the output
        // factor e^{(1-beta) M} Z'^{-beta} and the refusal; both halves then write O. The factor
        // is applied as two equal halves f = 2^{E/2}, O = (acc f) f, so that an output whose
        // value is within fp32 is not lost to a factor that alone overflows (or underflows).
        if (h == 1) s_zpart[r] = Zs + chk;  // chk is 0, or NaN to refuse
        ok = named_bar_and(kBarRows0 + (warp & 3), 64, ok && !*s_abort);
        if (h == 0) {
            Zs += s_zpart[r];
            bool bad = false;
            float f = 0.f;
            if (valid) {
                bad = isnan(chk) || !isfinite(M2) || !(Zs > 0.f) || !isfinite(Zs);
                const float E = (beta == 0.f) ? M2 : (1.f - beta) * M2 - beta * log2f(Zs);
                f = exp2f(0.5f * E);
            }
            if (__any_sync(0xffffffffu, bad) && lane == 0) flag_status(a.status, RS_STATUS_NONFINITE_BIT);
            s_zpart[r] = f;
        }
        // epilogue: every P V is in the accumulator once P V(diagonal) is done
        {
            const int t = numkv, sb = t % L::NSB;
            bool done = ok && wait_bar_warp(B.pv_done + sb, (t / L::NSB) & 1, s_abort, a.status);
            done = named_bar_and(kBarRows0 + (warp & 3), 64, done);  // also publishes f
            const float f = s_zpart[r];
            constexpr int nq = DVP / 32;  // 32-column chunks; half h writes chunks [h nq/2, (h+1) nq/2)
            if (done) {
                tc_fence_after();
                if (a.tma_out) {
                    // stage 128 rows x 32 columns per chunk in the free K/V ring, 16-byte units
                    // rotated by the row (r & 7) so that the row-wise writes here and the
                    // row-segment reads below both spread over all banks
                    const uint32_t stage_re = sbase + L::stages;
                    const uint32_t stage_im = stage_re + nq * kRegion;
#pragma unroll 1
                    for (int q = h * nq / 2; q < (h + 1) * nq / 2; ++q) {
                        uint32_t re[32], im[32];
                        RS_TMEM_LD32(trow + 32 * q, re);
                        if (GATED) RS_TMEM_LD32(trow + DVP + 32 * q, im);
                        tmem_ld_wait();
#pragma unroll
                        for (int c = 0; c < 8; ++c) {
                            const uint32_t off = q * kRegion + r * 128 + ((c ^ (r & 7)) << 4);
                            uint32_t wr[4], wi[4];
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const float xr = __uint_as_float(re[4 * c + k]);
                                wr[k] = __float_as_uint(xr == 0.f ? 0.f : (xr * f) * f);  // an exact 0 stays 0
                                if (GATED) {
                                    const float xi = __uint_as_float(im[4 * c + k]);
                                    wi[k] = __float_as_uint(xi == 0.f ? 0.f : (xi * f) * f);
                                }
                            }
                            sts128(stage_re + off, make_uint4(wr[0], wr[1], wr[2], wr[3]));
                            if (GATED) sts128(stage_im + off, make_uint4(wi[0], wi[1], wi[2], wi[3]));
                        }
                    }
                }
            }
            done = named_bar_and(kBarSoftmax, 256, done);
            if (done && a.tma_out) {
                // The staged chunks leave with coalesced 16-byte stores: lane l of each warp takes
                // 16-byte unit l % 8 of row l / 8 of a group of four rows, so one instruction
                // writes four whole 128-byte row segments. No copy engine is involved, so the CTA
                // need not wait for anything before it ends.
                const uint32_t stage_re = sbase + L::stages;
                const uint32_t stage_im = stage_re + nq * kRegion;
                const int wi = (tid - RL::sm_wg0 * 128) >> 5;  // 0..7 over both halves
                const int unit = lane & 7;
                const int nrows = min(128, n - sQ);
#pragma unroll 1
                for (int q = 0; q < nq; ++q) {
                    const int col = 32 * q + 4 * unit;
                    if (col >= a.dv) continue;  // dv % 4 == 0: whole 16-byte units
                    float *ore = a.O_re + (tok0 + sQ) * (int64_t)a.dv + col;
                    float *oim = a.O_im + (tok0 + sQ) * (int64_t)a.dv + col;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const int rr = 32 * k + 4 * wi + (lane >> 3);  // rows 0..127 over the 8 warps
                        if (rr >= nrows) continue;
                        const uint32_t off = q * kRegion + rr * 128 + ((unit ^ (rr & 7)) << 4);
                        const uint4 vr = lds128(stage_re + off);
                        *reinterpret_cast<uint4 *>(ore + (int64_t)rr * a.dv) = vr;
                        const uint4 vi = GATED ? lds128(stage_im + off) : make_uint4(0u, 0u, 0u, 0u);
                        *reinterpret_cast<uint4 *>(oim + (int64_t)rr * a.dv) = vi;
                    }
                }
            }
            if (done && !a.tma_out) {  // rows of dv % 4 != 0 floats: plain stores
                float *ore = a.O_re + (tok0 + row) * (int64_t)a.dv;
                float *oim = a.O_im + (tok0 + row) * (int64_t)a.dv;
#pragma unroll 1
                for (int q = h * nq / 2; q < (h + 1) * nq / 2; ++q) {
                    uint32_t re[32], im[32];
                    RS_TMEM_LD32(trow + 32 * q, re);  // warp-wide: every lane, valid row or not
                    if (GATED) RS_TMEM_LD32(trow + DVP + 32 * q, im);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (valid && 32 * q + e < a.dv) {
                            const float xr = __uint_as_float(re[e]);
                            const float xi = GATED ? __uint_as_float(im[e]) : 0.f;
                            ore[32 * q + e] = (xr == 0.f) ? 0.f : (xr * f) * f;
                            oim[32 * q + e] = (xi == 0.f) ? 0.f : (xi * f) * f;
                        }
                }
            }
        }
    }

    // ------------------------------------------------------------ teardown
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// Off-diagonal key tiles of each query tile of a table of gated heads: the key tiles run from
// KB = QB - 1 down and stop at the first one whose carry C(QB, KB) is exactly 0 (every
// farther tile is then exactly dead). One warp per query tile; the carries are scanned 32
// block totals at a time.
__global__ void __launch_bounds__(128)
head_numkv_kernel(HeadArgs a, const __grid_constant__ HeadTable tab)
{
    const int lane = threadIdx.x & 31;
    const int nqt = (a.n + 127) / 128;
    const int item = blockIdx.x * 4 + (threadIdx.x >> 5);
    if (item >= nqt * tab.count) return;
    const int slot = item / nqt, QB = item - slot * nqt;
    const float2 *T = a.carry + (int64_t)tab.bh[slot] * nqt;
    int numkv = QB;
    cplx run = {1.f, 0.f};
    for (int base = 0; base < QB; base += 32) {
        const int t = base + lane;
        cplx x = {1.f, 0.f};
        if (t < QB) {
            const float2 v = T[QB - 1 - t];
            x = {v.x, v.y};
        }
        cplx incl = x;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const cplx y = shfl_up(incl, d);
            if (lane >= d) incl = cmul(y, incl);
        }
        cplx excl = shfl_up(incl, 1);
        if (lane == 0) excl = {1.f, 0.f};
        const cplx Ct = cmul(run, excl);  // carry of tile t
        const unsigned z = __ballot_sync(0xffffffffu, t < QB && !cnonzero(Ct));
        if (z) {
            numkv = base + __ffs(z) - 1;
            break;
        }
        run = cmul(run, shfl_idx(incl, 31));
    }
    if (lane == 0) a.numkv[slot * nqt + QB] = numkv;
}

template <int DP, int DVP, bool GATED>
cudaError_t launch_t(const HeadArgs &a, const HeadTable &tab, const HeadMaps &maps, cudaStream_t s)
{
    using L = Cfg<DP, DVP, GATED>;
    auto k = head_fwd_kernel<DP, DVP, GATED>;
    // The register hand-over inside the kernel assumes the launch register count; a build
    // that came out smaller would make setmaxnreg.inc wait forever, so refuse to launch it.
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, k);
    if (e != cudaSuccess) return e;
    if (attr.numRegs < Roles<GATED>::launch_regs) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)L::alloc);
    if (e != cudaSuccess) return e;
    const int nqt = (a.n + 127) / 128;
    k<<<nqt * tab.count, Roles<GATED>::threads, L::alloc, s>>>(a, tab, maps);
    return cudaGetLastError();
}

template <bool GATED>
cudaError_t launch_g(const HeadArgs &a, const HeadTable &tab, const HeadMaps &maps, int dpad, int dvpad,
                     cudaStream_t s)
{
    if (dpad == 64 && dvpad == 64) return launch_t<64, 64, GATED>(a, tab, maps, s);
    if (dpad == 64 && dvpad == 128) return launch_t<64, 128, GATED>(a, tab, maps, s);
    if (dpad == 128 && dvpad == 64) return launch_t<128, 64, GATED>(a, tab, maps, s);
    return launch_t<128, 128, GATED>(a, tab, maps, s);
}

}  // namespace

cudaError_t launch_head_fwd(const HeadArgs &a, const HeadTable &tab, const HeadMaps &maps, int dpad, int dvpad,
                            cudaStream_t s)
{
    if (tab.count == 0 || a.n == 0) return cudaSuccess;
    // one launch serves heads of one kind: the caller splits gated and ungated heads
    return tab.g[0] != 0.f ? launch_g<true>(a, tab, maps, dpad, dvpad, s)
                           : launch_g<false>(a, tab, maps, dpad, dvpad, s);
}

cudaError_t launch_head_numkv(const HeadArgs &a, const HeadTable &tab, cudaStream_t s)
{
    if (tab.count == 0 || a.n == 0) return cudaSuccess;
    const int tiles = (a.n + 127) / 128 * tab.count;
    head_numkv_kernel<<<(tiles + 3) / 4, 128, 0, s>>>(a, tab);
    return cudaGetLastError();
}

}  // namespace rs
