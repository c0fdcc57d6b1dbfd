// head_common.cuh -- device helpers shared by the head kernels: bounded mbarrier waits,
// TMEM row loads, shared-memory vector access and accumulator row rescaling.
#pragma once

#include "gate_products.cuh"

namespace rs {
namespace head {

constexpr uint32_t kRegion = 128 * 128;   // one 128-row x 128-byte swizzled region (16 KB)
constexpr float kRescaleLog2 = 8.f;       // keep a stale maximum while the excess stays below 2^8

// Bounded wait on an mbarrier phase; also gives up when another role of this CTA (abort
// flag) or another CTA (status word) reported a timeout.
// Roles off the critical path pass sleep_ns > 0 and nap between polls, so that their
// spinning does not take issue slots from the softmax warps sharing their SM sub-partition.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort,
                                         int32_t *status, uint32_t sleep_ns = 0)
{
    const uint32_t addr = smem_u32(bar);
    if (mbar_try_wait(addr, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i) {
            if (mbar_try_wait(addr, parity)) return true;
            if (sleep_ns) __nanosleep(sleep_ns);
        }
        if (*abort) return false;
        if (*reinterpret_cast<volatile int32_t *>(status) & RS_STATUS_TIMEOUT_BIT) {
            *abort = 1;
            return false;
        }
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            flag_status(status, RS_STATUS_TIMEOUT_BIT);
            return false;
        }
    }
}

// The same, with one answer for the whole warp (the warp then stays converged for the
// warp-wide tcgen05.ld / tcgen05.st that follow).
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort,
                                              int32_t *status, uint32_t sleep_ns = 32)
{
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort, status, sleep_ns));
}

// Winding down. Whatever a CTA started must end before it frees TMEM and exits: TMA copies
// into its shared memory and tensor-core work on its TMEM and shared memory. After an abort
// nothing else waits for them, so the roles that started them do, with a time limit of
// their own that the abort flag does not cut short.
constexpr uint64_t kDrainLimitNs = 200000000ull;  // 0.2 s

// The TMA loads a producer issued into a ring of `nstages` stages with full barriers
// full[0 .. nstages): `issued` loads in order, load t into stage t % nstages. Waits for the
// phase of the last load of each stage (earlier phases of a barrier complete first).
__device__ __forceinline__ void drain_loads(uint64_t *full, int nstages, int issued)
{
    for (int s = 0; s < nstages && s < issued; ++s)
        mbar_wait(full + s, (uint32_t)((issued - 1 - s) / nstages) & 1u, kDrainLimitNs);
}

// Every tcgen05.mma this thread issued: a commit to `bar`, a barrier (count 1) that nothing
// else uses, and a wait for its first phase.
__device__ __forceinline__ void drain_mma(uint64_t *bar)
{
    umma_commit(bar);
    mbar_wait(bar, 0, kDrainLimitNs);
}

__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float (&v)[32])
{
    uint32_t r[32];
    RS_TMEM_LD32(taddr, r);
    tmem_ld_wait();
#pragma unroll
    for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
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

// acc row <- alpha * acc row (ncols fp32 columns)
__device__ __forceinline__ void scale_acc_row(uint32_t trow, int ncols, float alpha)
{
#pragma unroll 1
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

// (acc_re + i acc_im) <- z * (acc_re + i acc_im)
__device__ __forceinline__ void cscale_acc_row(uint32_t trow, int dvp, cplx z)
{
#pragma unroll 1
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

}  // namespace head
}  // namespace rs
