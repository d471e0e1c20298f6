// Launch helpers and programmatic dependent launch (opt-in).
//
// Every kernel of the library calls grid_dependency_sync() before it touches memory that
// an earlier kernel of the stream writes (and before nothing else: barrier setup and
// TMEM allocation may run early), then release_dependents().  Launched in plain stream
// order both return at once.  With programmatic dependent launch (the NSM_OPT_PDL
// option), kernels are launched with programmatic stream serialisation: the next
// kernel's launch and prologue then overlap the tail of the current one, and its own
// grid_dependency_sync() waits until this grid has completed and its writes are visible.
// Measured on one GB300, the overlap made the 4-matrix table 19% and the one-layer table
// 8% faster, but the GPT-2-small and Llama-7B tables 4.5% and 1.5% slower, so by
// default (auto) a call uses it only for tables of at most 2^25 elements.
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

inline bool pdl_enabled() { return pdl_for_launches(); }

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
