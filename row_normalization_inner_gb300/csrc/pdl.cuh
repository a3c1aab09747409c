// Programmatic dependent launch.  A kernel launched with
// launch_with_pdl may be scheduled before the kernel ahead of it in the
// stream has finished; it must call grid_dep_wait() before it reads or
// writes anything that kernel may touch (the wait returns once that kernel
// has completed and its memory is visible; with no programmatic predecessor
// it returns at once).  grid_dep_release() lets the next such launch be
// scheduled as soon as every CTA of this grid has executed it, so its CTAs
// take the SM slots this grid's last wave frees instead of waiting for the
// whole grid to drain.
#pragma once

#include <cuda_runtime.h>

namespace nf {

__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_release() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename Kernel, typename... Args>
cudaError_t launch_with_pdl(Kernel k, dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k, args...);
}

}  // namespace nf
