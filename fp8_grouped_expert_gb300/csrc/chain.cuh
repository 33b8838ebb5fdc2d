// Chains of programmatic dependent launches for the short kernels around the GEMMs (the
// routing kernels, the stacked prefill's glue).  A chained kernel starts with
// griddepcontrol.wait -- it touches nothing the kernel before it writes until that kernel
// has finished and its writes are visible, so results are those of plain stream order --
// and then lets its own dependent launch, so that launch overlaps this kernel instead of
// following its end.
#pragma once

#include <cuda_runtime.h>

namespace fge {

__device__ __forceinline__ void chain_enter() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launches kernel<<<grid, block, smem, s>>>(args...) as a programmatic dependent of the
// kernel before it on s.
template <typename... KArgs, typename... Args>
static cudaError_t launch_chained(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace fge
