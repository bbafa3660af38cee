// pdl.cuh -- programmatic dependent launch for the kernels of a decode step
// (cache write, decode, split merge: three launches on one stream).
//
// A kernel launched with the programmatic-serialization attribute may begin
// before the kernel ahead of it on the stream has finished, once every CTA
// of that kernel has called launch_dependents (or exited).  Each kernel here
// calls pdl_trigger() and then pdl_wait() before its first global-memory
// access: the wait returns only when the kernel ahead has completed and its
// writes are visible, so the only thing that overlaps is the launch and CTA
// placement of the next kernel with the tail of the current one.  Read-after-
// write (decode reads what the write stored; the merge reads the partials)
// and write-after-read (the next step's write over slots the decode read)
// both hold: a kernel completes only after its own wait has returned, so the
// chain of waits orders every kernel after all of its predecessors.  Without
// the attribute (PKV_PDL=0 in the environment, or a launch by other code)
// both instructions do nothing.
#pragma once

#include <cuda_runtime.h>

#include <cstdlib>
#include <utility>

namespace pkv {

__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// On unless PKV_PDL is set to a value starting with '0' (read once).
inline bool pdl_enabled() {
  static const bool on = [] {
    const char* e = std::getenv("PKV_PDL");
    return !(e != nullptr && e[0] == '0');
  }();
  return on;
}

// kernel<<<grid, block, smem, stream>>>(args...) with the programmatic-
// serialization attribute when enabled.
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

}  // namespace pkv
