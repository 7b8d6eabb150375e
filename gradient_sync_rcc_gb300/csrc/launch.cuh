// launch.cuh -- how every kernel of this library is launched: programmatic
// dependent launch (PDL) on the caller's stream.
//
// Device side: each kernel first waits for the grid ahead of it on the
// stream to complete and flush its memory (griddepcontrol.wait), before any
// global memory access, so stream order holds exactly as with a plain launch.
// Then it lets the next grid on the stream be scheduled as soon as all of its
// own CTAs have started (griddepcontrol.launch_dependents).  The next
// kernel's CTAs take the SM slots that this kernel's last wave frees and start
// the moment it completes, instead of after a fresh launch.  Launched without
// the attribute, or behind something other than a kernel, both instructions
// do nothing.
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>
#include <utility>

namespace rcc {

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait_then_release() {
  pdl_wait();
  pdl_release();
}

// RCC_PDL=0 launches without the attribute (plain stream order).
inline bool pdl_enabled() {
  static const bool on = [] {
    const char* v = std::getenv("RCC_PDL");
    return !(v && v[0] == '0');
  }();
  return on;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace rcc
