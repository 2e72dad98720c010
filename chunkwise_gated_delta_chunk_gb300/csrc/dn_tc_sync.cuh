// Synchronisation helpers of the tensor-core scan kernels (dn_tc.cu for
// dk = 128, dn_tc_wide.cu for dk = 256): bounded mbarrier waits with a shared
// abort flag, warp-uniform waits, the OR-reduction named barrier and the TMEM
// lane base of a warp.
//
// Every wait is bounded: after kTimeoutNs a CTA records kStatusTimeout in the
// status word and raises its abort flag, so that the other roles of the CTA
// stop too and drain their own outstanding copies and MMA work before the
// tensor memory is freed.
#pragma once

#include <stdint.h>

#include "dn_internal.h"
#include "tc_ptx.cuh"

namespace dn {
namespace tcs {
namespace {

constexpr uint64_t kTimeoutNs = kWaitLimitNs;

struct Ctx {
    uint32_t base;     // shared address of the aligned base
    uint8_t *gbase;    // generic pointer to the same
    volatile int *abort_flag;
    unsigned *status;
};

// Bounded wait.  Returns false once the CTA is aborting.
__device__ __noinline__ bool wait_slow(const Ctx &x, uint32_t b, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(b, parity)) return true;
        if ((it & 31u) == 0) {
            if (*x.abort_flag) return false;
            if (ptx::globaltimer() - t0 > kTimeoutNs) {
                *x.abort_flag = 1;
                atomicOr(x.status, kStatusTimeout);
                return false;
            }
        }
    }
}

__device__ __forceinline__ bool wait(const Ctx &x, uint32_t b, uint32_t parity) {
    if (ptx::mbar_try_wait(b, parity)) return true;
    return wait_slow(x, b, parity);
}

// Wait that ignores the abort flag (used while draining); bounded by time.
__device__ __noinline__ void wait_drain(uint32_t b, uint32_t parity) {
    const uint64_t t0 = ptx::globaltimer();
    while (!ptx::mbar_try_wait(b, parity))
        if (ptx::globaltimer() - t0 > kTimeoutNs) return;
}

// Warp-uniform wait: every lane gets the same answer, so lanes never diverge
// around the .sync.aligned tcgen05 instructions and warp syncs that follow.
__device__ __forceinline__ bool wwait(const Ctx &x, uint32_t b, uint32_t parity) {
    const bool ok = wait(x, b, parity);
    return __all_sync(0xffffffffu, ok);
}

// OR of `pred` over the `n` threads of named barrier `id` (also a barrier).
__device__ __forceinline__ bool bar_red_or(uint32_t id, uint32_t n, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// TMEM address of lane 32 (warp % 4), column 0: warp w reaches lanes
// 32 (w % 4) .. + 31, so each group of four consecutive warps covers all 128.
__device__ __forceinline__ uint32_t lane_base(uint32_t tmem, int warp) {
    return tmem + ((uint32_t)((warp & 3) * 32) << 16);
}

__device__ __forceinline__ void warp_arrive(uint32_t b) {
    __syncwarp();
    if ((threadIdx.x & 31) == 0) ptx::mbar_arrive(b);
}

}  // namespace
}  // namespace tcs
}  // namespace dn
