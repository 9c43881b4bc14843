// Programmatic dependent launch (PDL) helpers.
//
// Every kernel of the library is launched with programmatic stream
// serialization allowed: it may start while the previous kernel in the stream
// is still running, and it calls pdl_wait() before touching anything that
// kernel may write. pdl_wait() returns once the previous grid has completed
// and its memory is visible; pdl_trigger() (always after pdl_wait()) lets the
// next grid start. Since every kernel waits before it triggers, a kernel that
// starts has all kernels two or more launches back complete.
#pragma once
#include <cuda_runtime.h>

namespace moe {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
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
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace moe
