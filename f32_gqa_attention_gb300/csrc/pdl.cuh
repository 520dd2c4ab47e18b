// pdl.cuh -- programmatic dependent launch between consecutive launches of
// one call (CUDA's launch attribute and the griddepcontrol instructions of
// the PTX ISA).
//
// A kernel launched with launch_pdl may begin while the previous launch on
// the stream is still running: its CTAs are scheduled once every CTA of the
// previous launch has executed pdl_launch_dependents() (or exited), and each
// thread must call pdl_wait() -- which returns once the previous launch has
// completed and its memory writes are visible -- before its first access to
// anything that launch writes.  Work that does not depend on the previous
// launch (barrier set-up, descriptor prefetch, loads of the call's inputs)
// runs before the wait and overlaps the previous launch's tail.  In a kernel
// launched without the attribute both instructions do nothing.
#pragma once

#include <utility>

#include <cuda_runtime.h>

namespace vtmu {

__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

}  // namespace vtmu
