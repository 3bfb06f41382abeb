// Kernel launches with programmatic dependent launch (PDL).
//
// A step is a chain of kernels on one stream.  Every launch after the step's
// first carries cudaLaunchAttributeProgrammaticStreamSerialization, so the
// next kernel's CTAs may start (on SMs the previous kernel has left) and run
// their set-up before the previous kernel has finished.  Each kernel therefore
// executes grid_dependency_wait() in every CTA before it touches global memory
// that an earlier kernel of the step writes or reads; the wait returns once
// the previous grid has completed and its memory operations are visible.
// Because every CTA waits before it can exit, a kernel's completion implies
// its predecessor's, so dependencies on kernels further back hold too.
// allow_dependent_launch() lets the next kernel be scheduled early; it does
// not release any data.
#pragma once

#include <cuda_runtime.h>

#include <utility>

namespace muon {

__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// cudaLaunchKernelEx with the PDL attribute when `pdl` is set; returns the
// launch's cudaError_t as int.
template <typename... KArgs, typename... Args>
inline int launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, void* stream, bool pdl,
                         Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  if (pdl) {
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return (int)cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace muon
