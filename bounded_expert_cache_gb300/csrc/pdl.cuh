// Programmatic dependent launch for the decode chain (router, staging copy,
// gate/up, down): a kernel launched by pdl_launch may be scheduled while the
// previous kernel on the stream is still running. It calls pdl_wait() before
// it touches anything an earlier kernel writes (and before writing anything
// an earlier kernel reads), and pdl_trigger() right after, so at most its
// successor's prologue overlaps it. Kernels launched without the attribute
// return from both at once.
#pragma once

#include <cuda_runtime.h>

namespace moe {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... P, typename... A>
inline cudaError_t pdl_launch(void (*kernel)(P...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              A&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<A>(args)...);
}

}  // namespace moe
