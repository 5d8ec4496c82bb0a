// sync.cuh -- bounded mbarrier waits shared by the tcgen05 kernels.
//
// Every wait of a pipelined role is bounded: a wait that runs out raises the
// abort flag and BSA_ERR_TIMEOUT in the workspace and returns false, so the
// kernel drains its in-flight copies and MMAs, frees TMEM and exits cleanly.
#pragma once

#include <cstdint>

#include "internal.h"
#include "ptx.cuh"

namespace bsa {
namespace {

struct Ctl {
    volatile uint32_t *abort_flag;
    uint32_t *err;
    unsigned long long limit;
};

// Bounded wait on an mbarrier phase. Gives up (and raises the abort flag and
// BSA_ERR_TIMEOUT) after `limit` ns, or early when another role aborted.
__device__ __noinline__ bool wait_bar_slow(uint32_t bar, uint32_t parity, const Ctl &c)
{
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        // sleeps in hardware until the phase completes or ~50 us pass
        if (mbar_try_wait_sleep(bar, parity, 50000u)) return true;
        if (*c.abort_flag) return false;
        if (globaltimer_ns() - t0 > c.limit) {
            *c.abort_flag = 1u;
            raise_error(c.err, BSA_ERR_TIMEOUT);
            return false;
        }
    }
}

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl &c)
{
    return mbar_try_wait(bar, parity) || wait_bar_slow(bar, parity, c);
}

// Bounded wait used while draining in-flight async work on the way out; it
// ignores the abort flag.
__device__ __noinline__ bool wait_bar_drain(uint32_t bar, uint32_t parity, unsigned long long limit)
{
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait_sleep(bar, parity, 50000u))
        if (globaltimer_ns() - t0 > limit) return false;
    return true;
}

// Every lane waits (and acquires) itself; the verdict is made warp-uniform by a vote.
// (Cheaper than one lane waiting while the others park on a shuffle.)
__device__ __forceinline__ bool warp_wait_all(uint32_t bar, uint32_t parity, const Ctl &c)
{
    return __all_sync(0xffffffffu, wait_bar(bar, parity, c) ? 1 : 0) != 0;
}

}  // namespace
}  // namespace bsa
