// Kernel launch with programmatic stream serialization (internal helper of the library's launchers).
#pragma once
#include <cuda_runtime.h>

#include <utility>

namespace vd {

// Launches `kernel` so that it may begin while the previous kernel on `stream` is still finishing
// (programmatic dependent launch).  Every kernel of the library calls pdl_wait() before it touches
// global memory, so only its prologue (barrier set-up, tensor-memory allocation, descriptor
// prefetch) overlaps the previous kernel's tail.  Returns the launch error, if any.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace vd
