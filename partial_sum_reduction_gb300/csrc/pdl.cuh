// Programmatic dependent launch for the library's CUDA-core and collective
// kernels.  A kernel launched with launch_pdl is a programmatic dependent of
// the kernel before it in the stream: its CTAs may be placed on SMs that
// kernel frees, and wait in pdl_enter (its first statement) until that
// kernel has completed and its writes are visible.  pdl_enter then lets the
// next such kernel be scheduled.  SHMM_PDL=0 launches in plain stream order.
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>

namespace shmm_pdl {

__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    const char *e = getenv("SHMM_PDL");
    cfg.attrs = attr;
    cfg.numAttrs = (e && e[0] == '0') ? 0 : 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace shmm_pdl
