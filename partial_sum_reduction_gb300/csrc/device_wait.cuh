// Shared-memory mbarrier primitives and the bounded wait every pipeline wait
// of libshmm's kernels goes through.  A wait gives up after `limit` SM clock
// cycles: it raises the CTA's abort flag, records SHMM_ERR_TIMEOUT in the
// device status word and returns false, so the kernel can unwind (drain its
// own copies, free TMEM) and the host reads the failure with
// shmm_sync_status().  Nothing traps, nothing spins without a bound.
#pragma once

#include <cstdint>

#include "shmm.h"

namespace shmm_dev {

constexpr long long kWaitLimit = 4000000000LL;  // SM cycles (~2 s)

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait.  Returns false if the abort flag is raised (by this or
// another thread) or the wait outlives `limit` cycles, which raises it.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort_flag,
                                          int *status, bool honour_abort = true,
                                          long long limit = kWaitLimit) {
    long long t0 = 0;
    for (uint32_t it = 0;; ++it) {
        if (mbar_try(bar, parity)) return true;
        if (it == 0) t0 = clock64();
        if ((it & 31) == 31) {
            if (honour_abort && *abort_flag) return false;
            if (clock64() - t0 > limit) {
                *abort_flag = 1;
                atomicExch(status, (int)SHMM_ERR_TIMEOUT);
                return false;
            }
        }
    }
}

}  // namespace shmm_dev
