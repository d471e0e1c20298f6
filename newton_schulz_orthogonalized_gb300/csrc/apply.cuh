// The step's decay-and-update applied from a GEMM epilogue, shared by the grouped engine
// and the small-matrix kernel.  The update rule is the one of "DeepSpeed 集成 Muon 优化器实战"
// §核心算子: p <- p (1 - lr wd) - lr sqrt(max(1, rows/cols)) O, both terms on the old p.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "nsm_internal.h"

namespace nsm {
namespace {

// O's apply at natural positions (see ApplyArgs): o[j] is the stored-precision O at
// class (row, gc0 + j) of matrix mt.  Every load of the chunk is issued before its first
// store, so the 32 read-modify-writes of a lane overlap instead of queueing behind one
// another.
__device__ __forceinline__ void apply_chunk(const ApplyArgs& ap, const MatInfo& mt, int row, int gc0,
                                            int ncols, const float (&o)[32]) {
  float* __restrict__ p = ap.params + mt.off;
  __nv_bfloat16* __restrict__ pb =
      ap.params_bf16 ? reinterpret_cast<__nv_bfloat16*>(ap.params_bf16) + mt.off : nullptr;
  const float coef = ap.lr * mt.scale;
  const float decay = ap.decay;
  if (!mt.transposed && ncols == 32 && mt.vec_ok) {
    // class row = natural row: 32 consecutive parameters of this lane
    const int64_t i0 = static_cast<int64_t>(row) * mt.cols + gc0;
    float4* pp = reinterpret_cast<float4*>(p + i0);
    float4 a[8];
#pragma unroll
    for (int w = 0; w < 8; ++w) a[w] = pp[w];
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      a[w].x = fmaf(-coef, o[4 * w + 0], a[w].x * decay);
      a[w].y = fmaf(-coef, o[4 * w + 1], a[w].y * decay);
      a[w].z = fmaf(-coef, o[4 * w + 2], a[w].z * decay);
      a[w].w = fmaf(-coef, o[4 * w + 3], a[w].w * decay);
      pp[w] = a[w];
    }
    if (pb) {
      uint4* q = reinterpret_cast<uint4*>(pb + i0);
      const bool q16 = (reinterpret_cast<uintptr_t>(q) & 15) == 0;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        __nv_bfloat162 h[4] = {__floats2bfloat162_rn(a[2 * w].x, a[2 * w].y),
                               __floats2bfloat162_rn(a[2 * w].z, a[2 * w].w),
                               __floats2bfloat162_rn(a[2 * w + 1].x, a[2 * w + 1].y),
                               __floats2bfloat162_rn(a[2 * w + 1].z, a[2 * w + 1].w)};
        if (q16) {
          q[w] = *reinterpret_cast<const uint4*>(h);
        } else {
          __nv_bfloat162* q2 = reinterpret_cast<__nv_bfloat162*>(pb + i0 + 8 * w);
#pragma unroll
          for (int k = 0; k < 4; ++k) q2[k] = h[k];
        }
      }
    }
    return;
  }
  // general case: element (class row, gc0 + j) lives at natural (row, gc0 + j), or at
  // (gc0 + j, row) when the matrix is stored transposed in its class (then the lanes of
  // a warp cover consecutive natural columns)
  const int64_t step = mt.transposed ? mt.cols : 1;
  const int64_t i0 = mt.transposed ? static_cast<int64_t>(gc0) * mt.cols + row
                                   : static_cast<int64_t>(row) * mt.cols + gc0;
  float pv[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) pv[j] = j < ncols ? p[i0 + j * step] : 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j < ncols) {
      const float np = fmaf(-coef, o[j], pv[j] * decay);
      p[i0 + j * step] = np;
      if (pb) pb[i0 + j * step] = __float2bfloat16_rn(np);
    }
  }
}

}  // namespace
}  // namespace nsm
