// Index checks of the bounds-checked build (libshmm_checked.so, compiled
// with SHMM_CHECKED).  Each global load or store a kernel computes from its
// own index arithmetic first asks in_bounds() whether elements
// [first, first + count) lie inside the buffer's extent, which the launcher
// derives from the buffer sizes the interface documents, not from the
// kernel's loop bounds.  An index outside it records SHMM_ERR_BOUNDS in the
// device status word (shmm_sync_status reports it) and the access is
// skipped: nothing traps, nothing touches memory outside the buffer.  In the
// ordinary build in_bounds() is the constant true and the checks vanish.
#pragma once

#include <cstdint>

#include "shmm.h"

namespace shmm_dev {

__device__ __forceinline__ bool in_bounds(int *status, int64_t first, int64_t count, int64_t extent) {
#ifdef SHMM_CHECKED
    if (first >= 0 && count >= 0 && first <= extent - count) return true;
    if (status) atomicCAS(status, 0, (int)SHMM_ERR_BOUNDS);
    return false;
#else
    (void)status;
    (void)first;
    (void)count;
    (void)extent;
    return true;
#endif
}

}  // namespace shmm_dev
