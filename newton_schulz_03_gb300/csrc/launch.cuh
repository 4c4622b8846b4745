// launch.cuh -- programmatic dependent launch for the kernels of one step.
//
// Every kernel of the step is launched with programmatic stream
// serialisation: the next kernel in the stream may be scheduled while the
// previous one is still running, as soon as every CTA of the previous one
// has executed `griddepcontrol.launch_dependents`.  Its CTAs then set up
// (barriers, TMEM, tensor-map prefetch) and block in `griddepcontrol.wait`
// until the previous grid has completed and its memory is visible.  So a
// kernel must not read or write global memory before `grid_dep_wait()`.
// Launched without the attribute (or after a non-kernel stream operation)
// the wait returns at once and the launch is an ordinary serialised one.
//
// MUON_PDL=0 in the environment turns the attribute off (plain launches).
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <utility>

namespace muon {

__device__ __forceinline__ void grid_dep_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void grid_dep_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

inline bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("MUON_PDL");
    return !(v != nullptr && std::strcmp(v, "0") == 0);
  }();
  return on;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace muon
