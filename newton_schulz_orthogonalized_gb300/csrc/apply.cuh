// The step's decay-and-update applied from a GEMM epilogue, shared by the grouped engine
// and the small-matrix kernel.  The update rule is the one of "DeepSpeed 集成 Muon 优化器实战"
// §核心算子: p <- p (1 - lr wd) - lr sqrt(max(1, rows/cols)) O, both terms on the old p.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "nsm_internal.h"

namespace nsm {
namespace {

// O's apply at natural positions (see ApplyArgs).  A chunk is the 32 elements
// (row, gc0 + j), j < ncols, of matrix mt's class layout.  They live at natural
// (row, gc0 + j), or at (gc0 + j, row) when the matrix is stored transposed in its class;
// then the lanes of a warp cover consecutive natural columns.  apply_load reads the
// chunk's parameters and apply_store writes the updated ones, so a caller can issue the
// loads of the next chunk before the stores of this one.

// The 32 parameters of a wide matrix's row segment are 16-byte aligned and contiguous.
__device__ __forceinline__ bool apply_vec(const MatInfo& mt, int ncols) {
  return !mt.transposed && ncols == 32 && (mt.flags & kMatVec);
}

__device__ __forceinline__ void apply_load(const ApplyArgs& ap, const MatInfo& mt, int row, int gc0, int ncols,
                                           float (&pv)[32]) {
  const float* __restrict__ p = ap.params + mt.off;
  if (apply_vec(mt, ncols)) {
    const float4* pp = reinterpret_cast<const float4*>(p + static_cast<int64_t>(row) * mt.cols + gc0);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      const float4 a = pp[w];
      pv[4 * w + 0] = a.x;
      pv[4 * w + 1] = a.y;
      pv[4 * w + 2] = a.z;
      pv[4 * w + 3] = a.w;
    }
    return;
  }
  const int64_t step = mt.transposed ? mt.cols : 1;
  const int64_t i0 = mt.transposed ? static_cast<int64_t>(gc0) * mt.cols + row
                                   : static_cast<int64_t>(row) * mt.cols + gc0;
#pragma unroll
  for (int j = 0; j < 32; ++j) pv[j] = j < ncols ? p[i0 + j * step] : 0.f;
}

// p <- pv (1 - lr wd) - lr scale o, and its bf16 copy when requested.
__device__ __forceinline__ void apply_store(const ApplyArgs& ap, const MatInfo& mt, int row, int gc0, int ncols,
                                            const float (&o)[32], const float (&pv)[32]) {
  float* __restrict__ p = ap.params + mt.off;
  __nv_bfloat16* __restrict__ pb =
      ap.params_bf16 ? reinterpret_cast<__nv_bfloat16*>(ap.params_bf16) + mt.off : nullptr;
  const float coef = ap.lr * mt.scale;
  const float decay = ap.decay;
  if (apply_vec(mt, ncols)) {
    const int64_t i0 = static_cast<int64_t>(row) * mt.cols + gc0;
    float4* pp = reinterpret_cast<float4*>(p + i0);
    float np[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) np[j] = fmaf(-coef, o[j], pv[j] * decay);
#pragma unroll
    for (int w = 0; w < 8; ++w) pp[w] = make_float4(np[4 * w], np[4 * w + 1], np[4 * w + 2], np[4 * w + 3]);
    if (pb) {
      // i0 is a multiple of 8 elements and the copy is 16-byte aligned
      uint4* q = reinterpret_cast<uint4*>(pb + i0);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        __nv_bfloat162 h[4] = {__floats2bfloat162_rn(np[8 * w + 0], np[8 * w + 1]),
                               __floats2bfloat162_rn(np[8 * w + 2], np[8 * w + 3]),
                               __floats2bfloat162_rn(np[8 * w + 4], np[8 * w + 5]),
                               __floats2bfloat162_rn(np[8 * w + 6], np[8 * w + 7])};
        q[w] = *reinterpret_cast<const uint4*>(h);
      }
    }
    return;
  }
  const int64_t step = mt.transposed ? mt.cols : 1;
  const int64_t i0 = mt.transposed ? static_cast<int64_t>(gc0) * mt.cols + row
                                   : static_cast<int64_t>(row) * mt.cols + gc0;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j < ncols) {
      const float np = fmaf(-coef, o[j], pv[j] * decay);
      p[i0 + j * step] = np;
      if (pb) pb[i0 + j * step] = __float2bfloat16_rn(np);
    }
  }
}

__device__ __forceinline__ void apply_chunk(const ApplyArgs& ap, const MatInfo& mt, int row, int gc0,
                                            int ncols, const float (&o)[32]) {
  float pv[32];
  apply_load(ap, mt, row, gc0, ncols, pv);
  apply_store(ap, mt, row, gc0, ncols, o, pv);
}

}  // namespace
}  // namespace nsm
