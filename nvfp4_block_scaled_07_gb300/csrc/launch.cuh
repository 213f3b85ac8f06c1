// Host-side kernel launch with programmatic dependent launch (PDL).
//
// Every kernel of the library starts with griddepcontrol.wait before it
// touches global memory, and signals griddepcontrol.launch_dependents soon
// after, so a kernel launched here behind another kernel may be scheduled
// while its predecessor drains; its reads and writes still happen after the
// predecessor has completed.  NVFP4MOE_PDL=0 in the environment launches
// without the attribute (plain stream order), for comparisons.
#pragma once

#include <cstdlib>
#include <utility>

#include <cuda_runtime.h>

namespace nvfp4moe {

inline bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("NVFP4MOE_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                          bool cooperative, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  if (cooperative) {
    // A grid whose CTAs wait on one another: all of them resident at once.
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace nvfp4moe
