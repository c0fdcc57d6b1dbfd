// chain_scan.cu -- single-pass chunked forward substitution of (I - A) y = b (K3).
//
// "Resolvent Operator", section "The path-product corner is a resolvent": the readout at
// (beta, qk, g) = (0, 0, 1) is the chain y_i = a_i y_{i-1} + b_i, i.e. forward substitution
// of (I - A) y = b with A the gate shift. Here y_0 = b_0 (the page's y_0 = 0 is b_0 = 0).
//
// Each CTA takes a ticket (an atomic counter, so tickets follow the order CTAs start in)
// and owns one chunk of 128 tokens x dv channels of one head:
//   1. the chunk of b arrives in shared memory by one bulk copy; the gates are formed;
//   2. each of 8 warps runs the recurrence over its stretch of tokens (2 for warp 0, 18 for
//      the others) from a zero carry and keeps the affine map (A_w, Y_w) of its stretch:
//      y_out = A_w y_in + Y_w;
//   3. warp 0 composes the 8 maps into the chunk's map and hands it to warp 1, which
//      publishes it; meanwhile warp 0 looks back over earlier chunks of the same head (their
//      maps, or the carry a chunk already resolved) until it knows y at the end of the
//      previous chunk. A map with A = 0 (a closed gate) ends the look-back early;
//   4. every warp reruns its stretch from the true carry and writes y; warp 0 first
//      publishes the chunk's resolved carry.
// Publication is a release store of the chunk's flag after the data (a __syncwarp orders
// the other lanes' stores before it), and reading is an acquire load of the flag followed
// by a __syncwarp before the data loads; no other fence.
// b is read once and y written once. Every wait on another chunk is bounded in time and
// sets RS_STATUS_TIMEOUT (carry taken as 0) when it runs out, so the kernel always ends.
#include <mutex>

#include "common.cuh"

namespace rs {

namespace {

constexpr int kWarps = 8;
// Stretches: warp 0 takes 2 tokens and warps 1-7 take 18 each, because warp 0 also looks
// back and publishes the chunk's carry (whose release waits for its stores to complete)
// while the others run their stretches.
constexpr int kTok0 = 2, kTokW = 18;
static_assert(kTok0 + (kWarps - 1) * kTokW == kChainChunk, "stretches cover the chunk");
__device__ __forceinline__ int stretch_begin(int w) { return w == 0 ? 0 : kTok0 + (w - 1) * kTokW; }
constexpr int kBarMap = 1;  // named barrier: warp 0 hands the chunk's map to warp 1

__device__ __forceinline__ cplx to_cplx(float2 v) { return {v.x, v.y}; }

// Arrival without waiting (the producer side of a hand-off through shared memory: the
// barrier's completion orders this thread's earlier accesses before the waiting threads').
__device__ __forceinline__ void named_bar_arrive(int id, int count)
{
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

template <typename BT>
__device__ __forceinline__ float load_val(const BT *p);
template <>
__device__ __forceinline__ float load_val<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float load_val<__nv_bfloat16>(const __nv_bfloat16 *p)
{
    return __bfloat162float(*p);
}

// CTAs per SM that registers and shared memory both allow: six at dv <= 64, four at
// dv = 128 with bf16 b, three with fp32 b
template <int CPL, typename BT, bool NORM>
__global__ void __launch_bounds__(256, CPL <= 2 ? 6 : (sizeof(BT) == 2 ? 4 : 3))
chain_scan_kernel(ChainArgs a, const __grid_constant__ HeadTable tab)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ int s_ticket;
    __shared__ __align__(8) uint64_t s_bar;
    __shared__ cplx s_warpA[kWarps], s_exA[kWarps];
    // the normaliser chain z_i = m_i z_{i-1} + 1 (qk = 0 readout): warp maps
    __shared__ float s_wAz[kWarps], s_wYz[kWarps], s_exAz[kWarps], s_exYz[kWarps];
    __shared__ float s_zin;
    __shared__ cplx s_mapA;
    __shared__ float2 s_mapZ;

    const int dv = a.dv, n = a.n;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nchunks = (n + kChainChunk - 1) / kChainChunk;

    BT *sb = reinterpret_cast<BT *>(smem);                                     // [128][dv]
    cplx *s_warpY = reinterpret_cast<cplx *>(smem + sizeof(BT) * kChainChunk * dv);  // [8][dv]
    cplx *s_exY = s_warpY;  // the exclusive prefixes replace the warps' maps in place
    cplx *s_yin = s_warpY + kWarps * dv;                                        // [dv]
    // warp 0's exclusive prefix is the identity (never stored); its slot carries the chunk's
    // map from warp 0 to warp 1
    cplx *s_map = s_warpY;

    if (tid == 0) {
        s_ticket = atomicAdd(a.counter, 1);
        mbar_init(&s_bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    const int ticket = s_ticket;
    // chunk-major tickets: the heads of a table advance side by side, so each head has few
    // unresolved chunks in flight and look-backs stay short
    const int slot = ticket % tab.count, chunk = ticket / tab.count;
    if (chunk >= nchunks) return;
    const int64_t bh = tab.bh[slot];
    const float g = tab.g[slot];
    const int s0 = chunk * kChainChunk;
    const int len = min(kChainChunk, n - s0);
    const BT *bsrc = reinterpret_cast<const BT *>(a.b) + (bh * n + s0) * (int64_t)dv;
    const uint32_t bytes = (uint32_t)(len * dv * sizeof(BT));
    const bool bulk = (bytes % 16u) == 0 && (reinterpret_cast<uintptr_t>(bsrc) % 16u) == 0;

    if (bulk) {
        if (tid == 0) {
            mbar_arrive_expect_tx(&s_bar, bytes);
            bulk_load(sb, bsrc, bytes, &s_bar);
        }
    } else {
        for (int e = tid; e < len * dv; e += blockDim.x) sb[e] = bsrc[e];
    }

    // gates of this chunk ("Object": blended gate and gate): lane l of a warp holds the gate
    // of token l of its stretch (and its modulus) for the warp's two passes
    const int tok0 = stretch_begin(warp);
    const int ntok = warp == 0 ? kTok0 : kTokW;
    bool bad = false;
    cplx gate = {1.f, 0.f};
    float gmod = 1.f;
    if (lane < ntok) {
        const int t = s0 + tok0 + lane;
        cplx at = {1.f, 0.f};
        float mt = 1.f;
        if (tok0 + lane < len) {
            const float uu = a.u[bh * n + t], th = a.theta[bh * n + t];
            const float m = fminf(fmaxf(fmaf(g, uu, 1.f - g), 0.f), 1.f);
            const float tp = g * th;
            bad = !isfinite(uu) || !isfinite(th) || !isfinite(tp);
            float sn, cs;
            sincosf(tp, &sn, &cs);
            at = {m * cs, m * sn};
            mt = m;
            if (t == 0 && !a.carry_in) {  // y_0 = b_0 and z_0 = 1: nothing flows in ahead of token 0
                at = {0.f, 0.f};
                mt = 0.f;
            }
        }
        gate = at;
        gmod = mt;
    }
    if (__syncthreads_or(bad) && tid == 0) flag_status(a.status, RS_STATUS_NONFINITE_BIT);
    __shared__ int s_loaded;
    if (tid == 0) {
        s_loaded = !bulk || mbar_wait(&s_bar, 0, a.wait_limit_ns);
        if (!s_loaded) {
            flag_status(a.status, RS_STATUS_TIMEOUT_BIT);
            // the copy still lands in this CTA's shared memory: wait for it (with a limit of
            // its own) before the CTA exits
            mbar_wait(&s_bar, 0, 200000000ull);
        }
    }
    __syncthreads();
    if (!s_loaded) return;  // the chunk never arrived: give up on it (uniform across the CTA)

    const int ch0 = lane * CPL;
    const int tok1 = min(tok0 + ntok, len);

    // pass 1: each warp's stretch as an affine map from a zero carry
    {
        cplx y[CPL];
        cplx A = {1.f, 0.f};
#pragma unroll
        for (int c = 0; c < CPL; ++c) y[c] = {0.f, 0.f};
        for (int t = tok0; t < tok1; ++t) {
            const cplx at = shfl_idx(gate, t - tok0);
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const float bv = (ch0 + c < dv) ? load_val(sb + t * dv + ch0 + c) : 0.f;
                y[c] = cmul(at, y[c]);
                y[c].re += bv;
            }
            A = cmul(at, A);
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c)
            if (ch0 + c < dv) s_warpY[warp * dv + ch0 + c] = y[c];
        if (lane == 0) s_warpA[warp] = A;
        if (NORM) {  // the same stretch of the real chain (every lane alike)
            float Az = 1.f, Yz = 0.f;
            for (int t = tok0; t < tok1; ++t) {
                const float m = __shfl_sync(0xffffffffu, gmod, t - tok0);
                Yz = fmaf(m, Yz, 1.f);
                Az *= m;
            }
            if (lane == 0) {
                s_wAz[warp] = Az;
                s_wYz[warp] = Yz;
            }
        }
    }
    __syncthreads();

    // warp 0: the chunk's map (eA, eY; eAz, eYz for the normaliser) and the carry into the
    // chunk (yin, zin)
    cplx eA = {1.f, 0.f};
    cplx eY[CPL], yin[CPL];
#pragma unroll
    for (int c = 0; c < CPL; ++c) eY[c] = yin[c] = {0.f, 0.f};
    float eAz = 1.f, eYz = 0.f, zin = 0.f;
    const int64_t me = (int64_t)slot * nchunks + chunk;
    const bool publish = ticket != a.withhold_chunk;
    if (warp == 0) {
        // compose the warps' maps: exclusive prefixes and the chunk's map
        for (int w = 0; w < kWarps; ++w) {
            if (lane == 0) s_exA[w] = eA;
            const cplx wA = s_warpA[w];
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                // each lane reads its channels of warp w's map, then overwrites them with the
                // exclusive prefix
                const cplx wY = (ch0 + c < dv) ? s_warpY[w * dv + ch0 + c] : cplx{0.f, 0.f};
                if (ch0 + c < dv) s_exY[w * dv + ch0 + c] = eY[c];
                const cplx t = cmul(wA, eY[c]);
                eY[c] = {t.re + wY.re, t.im + wY.im};
            }
            eA = cmul(wA, eA);
        }
        if (NORM) {
            for (int w = 0; w < kWarps; ++w) {
                if (lane == 0) {
                    s_exAz[w] = eAz;
                    s_exYz[w] = eYz;
                }
                eYz = fmaf(s_wAz[w], eYz, s_wYz[w]);
                eAz *= s_wAz[w];
            }
        }
        if (chunk > 0 && publish) {
            // warp 1 publishes the chunk's map while this warp looks back
#pragma unroll
            for (int c = 0; c < CPL; ++c)
                if (ch0 + c < dv) s_map[ch0 + c] = eY[c];
            if (lane == 0) {
                s_mapA = eA;
                s_mapZ = make_float2(eAz, eYz);
            }
            named_bar_arrive(kBarMap, 64);
        }
        if (chunk == 0) {
            // before the first chunk: the carry of the previous segment, or nothing
            if (a.carry_in) {
#pragma unroll
                for (int c = 0; c < CPL; ++c)
                    if (ch0 + c < dv) yin[c] = to_cplx(a.carry_in[bh * dv + ch0 + c]);
            }
        } else {
            // look back: acc maps y_end(p) to y_end(chunk-1) (and z likewise)
            float accAz = 1.f, accYz = 0.f;
            cplx accA = {1.f, 0.f};
            cplx accY[CPL];
#pragma unroll
            for (int c = 0; c < CPL; ++c) accY[c] = {0.f, 0.f};
            for (int p = chunk - 1; p >= 0; --p) {
                const int64_t other = (int64_t)slot * nchunks + p;
                int f = lane == 0 ? ld_acquire_gpu(a.flags + other) : 0;
                f = __shfl_sync(0xffffffffu, f, 0);
                if (f == 0) {
                    if (lane == 0) {
                        const uint64_t t0 = globaltimer_ns();
                        while ((f = ld_acquire_gpu(a.flags + other)) == 0) {
                            if (globaltimer_ns() - t0 > a.wait_limit_ns) break;
                            __nanosleep(64);
                        }
                    }
                    f = __shfl_sync(0xffffffffu, f, 0);
                }
                // lane 0's acquire, then __syncwarp: the other lanes' loads below come after it
                __syncwarp();
                if (f == 0) {  // ran out of time: take the carry as 0 and say so
                    if (lane == 0) flag_status(a.status, RS_STATUS_TIMEOUT_BIT);
#pragma unroll
                    for (int c = 0; c < CPL; ++c) yin[c] = accY[c];
                    zin = accYz;
                    break;
                }
                if (f == 2) {
#pragma unroll
                    for (int c = 0; c < CPL; ++c) {
                        cplx yp = {0.f, 0.f};
                        if (ch0 + c < dv) {
                            const float2 v = __ldcg(a.incl_y + other * dv + ch0 + c);
                            yp = {v.x, v.y};
                        }
                        const cplx t = cmul(accA, yp);
                        yin[c] = {t.re + accY[c].re, t.im + accY[c].im};
                    }
                    if (NORM) zin = fmaf(accAz, __ldcg(a.incl_z + other), accYz);
                    break;
                }
                const float2 pa = __ldcg(a.agg_a + other);
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    cplx yp = {0.f, 0.f};
                    if (ch0 + c < dv) {
                        const float2 v = __ldcg(a.agg_y + other * dv + ch0 + c);
                        yp = {v.x, v.y};
                    }
                    const cplx t = cmul(accA, yp);
                    accY[c] = {t.re + accY[c].re, t.im + accY[c].im};
                }
                accA = cmul(accA, {pa.x, pa.y});
                if (NORM) {
                    const float2 pz = __ldcg(a.agg_z + other);
                    accYz = fmaf(accAz, pz.y, accYz);
                    accAz *= pz.x;
                }
                if (!cnonzero(accA)) {  // a closed gate: nothing earlier reaches this chunk
#pragma unroll
                    for (int c = 0; c < CPL; ++c) yin[c] = accY[c];
                    zin = accYz;
                    break;
                }
            }
        }
#pragma unroll
        for (int c = 0; c < CPL; ++c)
            if (ch0 + c < dv) s_yin[ch0 + c] = yin[c];
        if (lane == 0) s_zin = zin;
    } else if (warp == 1 && chunk > 0 && publish) {
        // the chunk's map (flag 1), so that later chunks can look past this one before its
        // carry is resolved; __syncwarp orders every lane's stores before lane 0's release
        named_bar_sync(kBarMap, 64);
#pragma unroll
        for (int c = 0; c < CPL; ++c)
            if (ch0 + c < dv) {
                const cplx m = s_map[ch0 + c];
                a.agg_y[me * dv + ch0 + c] = make_float2(m.re, m.im);
            }
        if (lane == 0) {
            a.agg_a[me] = make_float2(s_mapA.re, s_mapA.im);
            if (NORM) a.agg_z[me] = s_mapZ;
        }
        __syncwarp();
        if (lane == 0) st_release_gpu(a.flags + me, 1);
    }
    __syncthreads();
    // the resolved carry y_end(chunk) = eA y_in + eY, published after the barrier: the
    // release waits for warp 0's stores to complete, and the other warps write y meanwhile
    if (warp == 0 && publish) {
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            const cplx t = cmul(eA, yin[c]);
            if (ch0 + c < dv)
                a.incl_y[me * dv + ch0 + c] = make_float2(t.re + eY[c].re, t.im + eY[c].im);
        }
        if (NORM && lane == 0) a.incl_z[me] = fmaf(eAz, zin, eYz);
        // __syncwarp orders every lane's stores before lane 0's release of the flag
        __syncwarp();
        if (lane == 0) st_release_gpu(a.flags + me, 2);
    }

    // pass 2: rerun each stretch from its true carry and write y
    {
        const cplx wA = s_exA[warp];
        cplx y[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) {
            if (ch0 + c < dv) {
                const cplx t = cmul(wA, s_yin[ch0 + c]);
                const cplx e = warp == 0 ? cplx{0.f, 0.f} : s_exY[warp * dv + ch0 + c];
                y[c] = {t.re + e.re, t.im + e.im};
            } else {
                y[c] = {0.f, 0.f};
            }
        }
        float *yr = a.y_re + (bh * n + s0) * (int64_t)dv;
        float *yi = a.y_im + (bh * n + s0) * (int64_t)dv;
        // qk = 0 readout: O_i = y_i z_i^{-beta}
        const float beta = tab.beta[slot];
        const bool scale_out = NORM && beta != 0.f;
        // z_i = m_i z_{i-1} + 1 at each token of the stretch: lane l composes the maps
        // x -> m x + 1 of tokens tok0 .. tok0 + l (a warp scan), applies them to z at the end of
        // the previous stretch, and works out its token's factor z^{-beta} once
        float fz_lane = 1.f;
        if (scale_out) {
            const bool mine = lane < tok1 - tok0;
            float A = mine ? gmod : 1.f, Bz = mine ? 1.f : 0.f;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const float Ap = __shfl_up_sync(0xffffffffu, A, d), Bp = __shfl_up_sync(0xffffffffu, Bz, d);
                if (lane >= d) {
                    Bz = fmaf(A, Bp, Bz);
                    A *= Ap;
                }
            }
            const float zl = fmaf(A, fmaf(s_exAz[warp], s_zin, s_exYz[warp]), Bz);
            fz_lane = exp2f(-beta * log2f(zl));
        }
        for (int t = tok0; t < tok1; ++t) {
            const cplx at = shfl_idx(gate, t - tok0);
            float vr[CPL], vi[CPL];
            const bool last = a.carry_out && s0 + t == n - 1;
            const float fz = scale_out ? __shfl_sync(0xffffffffu, fz_lane, t - tok0) : 1.f;
#pragma unroll
            for (int c = 0; c < CPL; ++c) {
                const float bv = (ch0 + c < dv) ? load_val(sb + t * dv + ch0 + c) : 0.f;
                y[c] = cmul(at, y[c]);
                y[c].re += bv;
                vr[c] = y[c].re * fz;
                vi[c] = y[c].im * fz;
                if (last && ch0 + c < dv) a.carry_out[bh * dv + ch0 + c] = make_float2(y[c].re, y[c].im);
            }
            if (ch0 + CPL <= dv && (dv % CPL) == 0) {
                if constexpr (CPL == 4) {
                    *reinterpret_cast<float4 *>(yr + t * dv + ch0) = make_float4(vr[0], vr[1], vr[2], vr[3]);
                    *reinterpret_cast<float4 *>(yi + t * dv + ch0) = make_float4(vi[0], vi[1], vi[2], vi[3]);
                } else if constexpr (CPL == 2) {
                    *reinterpret_cast<float2 *>(yr + t * dv + ch0) = make_float2(vr[0], vr[1]);
                    *reinterpret_cast<float2 *>(yi + t * dv + ch0) = make_float2(vi[0], vi[1]);
                } else {
                    yr[t * dv + ch0] = vr[0];
                    yi[t * dv + ch0] = vi[0];
                }
            } else {
#pragma unroll
                for (int c = 0; c < CPL; ++c)
                    if (ch0 + c < dv) {
                        yr[t * dv + ch0 + c] = vr[c];
                        yi[t * dv + ch0 + c] = vi[c];
                    }
            }
        }
    }
}

template <int CPL, typename BT, bool NORM>
cudaError_t launch_t(const ChainArgs &a, const HeadTable &tab, cudaStream_t s)
{
    const int nchunks = (a.n + kChainChunk - 1) / kChainChunk;
    const size_t smem = sizeof(BT) * kChainChunk * a.dv + sizeof(cplx) * (kWarps + 1) * a.dv;
    auto k = chain_scan_kernel<CPL, BT, NORM>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // all of the SM's unified L1 / shared memory as shared memory: six CTAs of 128 tokens x 64
    // fp32 channels fit
    e = cudaFuncSetAttribute(k, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return e;
    k<<<tab.count * nchunks, 256, smem, s>>>(a, tab);
    return cudaGetLastError();
}

}  // namespace

// Scratch of resolvent_chain_scan_noalloc: one fixed array in device memory, reserved when
// the library's device code is loaded in a context (with lazy module loading, at the first
// call that needs it) and held until the process exits. Host code must not pass
// `g_chain_noalloc_scratch` itself to a kernel (on the host it names a stand-in, not a
// device address); chain_noalloc_scratch() looks up the device address once per device and
// context: a context made after cudaDeviceReset holds a new copy of the array, so the
// address is looked up again when the current context's id changes.
static __device__ __align__(256) unsigned char g_chain_noalloc_scratch[kChainNoAllocBytes];

namespace {
// cuCtxGetId through the runtime's driver entry point (no link against libcuda)
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
bool current_context_id(unsigned long long *id)
{
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    CUcontext ctx = nullptr;
    if (!get_current || !get_id || get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}
}  // namespace

cudaError_t chain_noalloc_scratch(void **ptr)
{
    constexpr int kMaxDevices = 64;
    static void *addr[kMaxDevices] = {};
    static unsigned long long ctx_of[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    // cudaSetDevice makes the device's primary context current (creating it on first use),
    // so that its id can be read before the first launch
    e = cudaSetDevice(dev);
    if (e != cudaSuccess) return e;
    unsigned long long ctx = 0;
    if (!current_context_id(&ctx)) return cudaErrorDeviceUninitialized;
    std::lock_guard<std::mutex> lk(mu);
    if (!addr[dev] || ctx_of[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_chain_noalloc_scratch);  // with `dev` current
        if (e != cudaSuccess) return e;
        addr[dev] = p;
        ctx_of[dev] = ctx;
    }
    *ptr = addr[dev];
    return cudaSuccess;
}

size_t chain_scratch_bytes(int slots, int n, int dv)
{
    const size_t nchunks = (size_t)(n + kChainChunk - 1) / kChainChunk;
    const size_t chunks = (size_t)slots * nchunks;
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return up(sizeof(int) * (chunks + 1)) + up(sizeof(float2) * chunks) +
           2 * up(sizeof(float2) * chunks * (size_t)dv) + up(sizeof(float2) * chunks) +
           up(sizeof(float) * chunks);
}

template <bool NORM>
cudaError_t launch_n(const ChainArgs &a, const HeadTable &tab, cudaStream_t s)
{
    if (a.dv <= 32) return a.b_is_bf16 ? launch_t<1, __nv_bfloat16, NORM>(a, tab, s) : launch_t<1, float, NORM>(a, tab, s);
    if (a.dv <= 64) return a.b_is_bf16 ? launch_t<2, __nv_bfloat16, NORM>(a, tab, s) : launch_t<2, float, NORM>(a, tab, s);
    return a.b_is_bf16 ? launch_t<4, __nv_bfloat16, NORM>(a, tab, s) : launch_t<4, float, NORM>(a, tab, s);
}

cudaError_t launch_chain_scan(const ChainArgs &a, const HeadTable &tab, cudaStream_t s)
{
    if (tab.count == 0 || a.n == 0) return cudaSuccess;
    // the normaliser chain is compiled only into the qk = 0 readout variant
    return a.normalize ? launch_n<true>(a, tab, s) : launch_n<false>(a, tab, s);
}

}  // namespace rs
