// device_common.cuh - bounded mbarrier waits shared by the kernels.
//
// Every wait in the kernels is bounded: after `timeout_ns` of %globaltimer time the
// waiting thread records an error code in the per-device error word, raises the CTA's
// abort flag (so the other roles stop waiting too) and returns false.  Nothing traps;
// the kernel drains its in-flight copies and MMAs, frees its tensor memory and exits,
// and the host reads the code with gsr_device_status().
#pragma once

#include "kernels.h"
#include "ptx.cuh"

namespace gsr {

struct Waiter {
    int* err;                       // device error word (first code wins)
    uint64_t timeout_ns;
    volatile uint32_t* abort_flag;  // shared memory, one per CTA
    int kernel_code;                // kDevErrKernelTiled / kDevErrKernelSkinny

    __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity, int code) const {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t spin = 1;; ++spin) {
            if (mbar_try_wait(bar, parity)) return true;
            if ((spin & 63u) == 0u) {
                if (*abort_flag) return false;
                if (globaltimer_ns() - t0 > timeout_ns) {
                    *abort_flag = 1u;
                    atomicCAS(err, 0, kernel_code | code);
                    return false;
                }
            }
        }
    }

    // Teardown variant: ignores the abort flag (it must really drain), still bounded.
    __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
        if (mbar_try_wait(bar, parity)) return true;
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t spin = 1;; ++spin) {
            if (mbar_try_wait(bar, parity)) return true;
            if ((spin & 63u) == 0u && globaltimer_ns() - t0 > timeout_ns) {
                *abort_flag = 1u;
                atomicCAS(err, 0, kernel_code | kDevErrTeardown);
                return false;
            }
        }
    }

    __device__ __forceinline__ bool aborted() const { return *abort_flag != 0u; }
};

}  // namespace gsr
