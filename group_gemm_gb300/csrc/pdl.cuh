// pdl.cuh -- programmatic dependent launch for every kernel of the library.
//
// A kernel launched with programmatic stream serialization may begin while the kernel before it
// on the stream is still running: its CTAs take the SMs that kernel has already left, set up what
// touches no global memory (barriers, tensor memory, prefetch of tensor maps passed as
// parameters), and only then wait until the previous grid has completed and its writes are
// visible (griddepcontrol.wait). Every kernel here also signals at its start that the next one
// may be scheduled (griddepcontrol.launch_dependents): that kernel's CTAs still find room only
// on SMs this one has left, and they wait the same way, so a chain of launches never runs ahead
// of its data. Between launches this hides the launch latency and the prologue of the next
// kernel behind the tail of the previous one.
#pragma once

#include <cuda_runtime.h>

namespace rdot {

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void grid_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Start of a kernel that has no set-up to overlap: let the next kernel be scheduled, then wait
// for the previous one.
__device__ __forceinline__ void grid_dependency_enter() {
    grid_launch_dependents();
    grid_dependency_wait();
}

// kern<<<grid, block, shm, stream>>>(args...) with programmatic stream serialization allowed.
// Cluster dimensions declared on the kernel (__cluster_dims__) apply as with <<<>>>.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t shm, cudaStream_t stream,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = shm;
    cfg.stream = stream;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

}  // namespace rdot
