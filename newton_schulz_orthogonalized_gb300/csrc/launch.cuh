// Launch helpers and programmatic dependent launch (opt-in).
//
// Every kernel of the library calls grid_dependency_sync() before it touches memory that
// an earlier kernel of the stream writes (and before nothing else: barrier setup and
// TMEM allocation may run early), then release_dependents().  Launched in plain stream
// order (the default) both return at once.  With the NSM_OPT_PDL option set, kernels
// are launched with programmatic stream serialisation: the next kernel's launch and
// prologue then overlap the tail of the current one, and its own grid_dependency_sync()
// waits until this grid has completed and its writes are visible.  Measured on one
// GB300, the overlap made the 4-matrix table 13% faster (0.066 -> 0.058 ms) but the
// GPT-2-small and Llama-7B tables 6-9% and 1.5% slower, so it is off by default.
#pragma once

#include <cuda_runtime.h>

#include "nsm_internal.h"

namespace nsm {

__device__ __forceinline__ void grid_dependency_sync() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}

__device__ __forceinline__ void release_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

inline bool pdl_enabled() { return option_value(NSM_OPT_PDL) != 0; }

// `overlap` = false launches in plain stream order (the kernel's own dependency sync then
// returns at once).
template <typename... KArgs, typename... Args>
cudaError_t launch_ordered(bool overlap, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                           cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = (overlap && pdl_enabled()) ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args) {
  return launch_ordered(true, kernel, grid, block, smem, stream, args...);
}

}  // namespace nsm
