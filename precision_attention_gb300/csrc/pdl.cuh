// pdl.cuh -- programmatic dependent launch between the step's kernels.
//
// A kernel launched with launch_pdl may be scheduled while the kernel before it
// in the stream is still running, once that kernel has executed pdl_trigger()
// in every CTA (or has finished). It must call pdl_wait() before it reads
// anything the previous kernel writes and before it overwrites anything the
// previous kernel reads; pdl_wait() returns once the previous kernel has
// completed and its memory operations are visible. A kernel whose completion
// must imply its predecessor's (so that the next kernel's pdl_wait() covers
// both) calls pdl_wait() before it exits. Without the launch attribute both
// instructions do nothing, and a CUDA graph capture keeps the dependencies as
// programmatic edges.
#pragma once
#include <cuda_runtime.h>

#include <utility>

namespace pa {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <class... KArgs, class... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
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
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace pa
