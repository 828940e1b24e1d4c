// watchdog.cuh -- bounded mbarrier waits.
//
// Every pipeline wait in libhgemm goes through these.  A wait gives up when
// (a) the phase completes (success), (b) another role of the same CTA has
// already given up (the CTA-shared abort flag), or (c) its own deadline on
// %globaltimer passes, or an iteration cap is hit.  In case (c) it records an
// error code in the plan's device error word (first error wins), raises the
// abort flag, and returns false; the caller then skips to teardown: it waits,
// again with a deadline, for its own copies and MMAs in flight, frees its TMEM
// and returns.  No wait can spin forever and no error path traps.
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace hg {

// Error word layout: bit 31 set = a wait timed out; bits 16-23 = role;
// bits 0-15 = barrier index within that role.
enum : uint32_t {
    ROLE_PRODUCER = 1,
    ROLE_MMA = 2,
    ROLE_EPILOGUE = 3,
    ROLE_DRAIN = 4,
    ROLE_SELFTEST = 5,
};

__host__ __device__ constexpr int32_t timeout_code(uint32_t role, uint32_t index) {
    return static_cast<int32_t>(0x80000000u | (role << 16) | (index & 0xFFFFu));
}

// Invariant violations (debug checks): bit 30 set; bits 16-23 the kernel
// (KERNEL_*), bits 0-15 which check failed.
enum : uint32_t { KERNEL_TILED = 1, KERNEL_PAIR = 2, KERNEL_SKINNY = 3 };
enum : uint32_t {
    CHECK_TILE = 1,   // tile index or its (batch, m, n) outside the output
    CHECK_KRANGE = 2, // K range empty or outside K
    CHECK_PIECE = 3,  // piece / segment index outside its tile's pieces
};
__host__ __device__ constexpr int32_t invariant_code(uint32_t kernel, uint32_t check) {
    return static_cast<int32_t>(0x40000000u | (kernel << 16) | (check & 0xFFFFu));
}

// Records a failed invariant (first error wins) and reports it to the caller,
// who stops before using the work item.
__device__ __forceinline__ bool invariant_failed(int32_t *err, int32_t code) {
    atomicCAS(err, 0, code);
    return false;
}

// Hard cap on polling iterations, independent of the clock.
constexpr uint32_t kMaxWaitIterations = 1u << 30;
// mbarrier polls between two reads of the clock and the abort flag.
constexpr int kPollsPerCheck = 16;

struct WaitCtl {
    volatile int32_t *abort_flag;  // shared memory, CTA scope
    int32_t *err;                  // device error word (global memory)
    uint64_t timeout_ns;
};

// Single-thread bounded wait.  `honor_abort == false` is used on teardown,
// where a thread must still wait for its own operations after an abort.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity, const WaitCtl &c,
                                             int32_t code, bool honor_abort = true) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 0; it < kMaxWaitIterations; ++it) {
        // several polls per clock and abort check: those reads would
        // otherwise dominate the loop and delay seeing the phase complete
#pragma unroll 1
        for (int k = 0; k < kPollsPerCheck; ++k)
            if (mbar_try_wait(bar, parity)) return true;
        if (honor_abort && *c.abort_flag) return false;
        if (globaltimer_ns() - t0 > c.timeout_ns) break;
    }
    if (honor_abort) {
        atomicCAS(c.err, 0, code);
        *c.abort_flag = 1;
    }
    return false;
}

// Whole-warp bounded wait with a warp-uniform result.  Lane 0 polls; on
// success every lane performs one (immediately satisfied) try_wait of its own
// so that each lane acquires the barrier's release.
__device__ __forceinline__ bool wait_bounded_warp(uint32_t bar, uint32_t parity, const WaitCtl &c,
                                                  int32_t code) {
    const uint32_t lane = threadIdx.x & 31u;
    int ok = 0;
    if (lane == 0) ok = wait_bounded(bar, parity, c, code) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (ok) (void)mbar_try_wait(bar, parity);
    __syncwarp();
    return ok != 0;
}

}  // namespace hg
