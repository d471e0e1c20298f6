// The step's decay-and-update applied from a kernel epilogue, shared by the grouped GEMM
// engine and the small-matrix kernel.  The update rule is the one of "DeepSpeed 集成 Muon 优化器实战"
// §核心算子: p <- p (1 - lr wd) - lr sqrt(max(1, rows/cols)) O, both terms on the old p.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cstdint>

#include "nsm_internal.h"

namespace nsm {
namespace {

// ---- 32 x 32 blocks, one natural column per lane (coalesced) -----------------------
//
// The block of class rows [rb, rb + 32) and class columns [gc0, gc0 + 32) of matrix mt
// covers natural rows r0 + j (j < nr) and natural columns c0 + lane (lane < nc): a tall
// matrix sits transposed in its class, so its class row rb + lane is natural column
// rb + lane; for a wide one the block is transposed.  Every load and store of a warp is
// then one 128-byte access.
struct ApplyBlock {
  int r0, c0, nr, nc;
};

__device__ __forceinline__ ApplyBlock apply_block_at(const MatInfo& mt, int rb, int gc0, int class_rows,
                                                     int class_cols) {
  const int in_cols = min(32, class_cols - gc0), in_rows = min(32, class_rows - rb);
  if (mt.transposed) return {gc0, rb, in_cols, in_rows};
  return {rb, gc0, in_rows, in_cols};
}

__device__ __forceinline__ void apply_block_load(const ApplyArgs& ap, const MatInfo& mt, const ApplyBlock& k,
                                                 int lane, float (&pv)[32]) {
  const int64_t cols = mt.cols;
  const float* src = ap.params + mt.off + static_cast<int64_t>(k.r0) * cols + k.c0 + lane;
#pragma unroll
  for (int j = 0; j < 32; ++j) pv[j] = (j < k.nr && lane < k.nc) ? src[j * cols] : 0.f;
}

// Puts element j of the lane's natural column into o[j/2] (half j & 1): for a wide matrix
// the lane's class row (packed pairs in o) is transposed through xw (32 rows x 17 words
// of this warp's shared memory).
__device__ __forceinline__ void apply_block_columns(const MatInfo& mt, uint32_t (&o)[16], uint32_t* xw, int lane) {
  if (mt.transposed) return;
#pragma unroll
  for (int i = 0; i < 16; ++i) xw[lane * 17 + i] = o[i];
  __syncwarp();
  const int wc = lane >> 1;
  const uint32_t sel = (lane & 1) ? 0x7632u : 0x5410u;
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i] = __byte_perm(xw[(2 * i) * 17 + wc], xw[(2 * i + 1) * 17 + wc], sel);
  __syncwarp();
}

// p <- pv (1 - lr wd) - lr scale o over the block (o: stored 16-bit values, FP16 selects
// fp16 or bf16), and the bf16 copy when requested.
template <bool FP16>
__device__ __forceinline__ void apply_block_store(const ApplyArgs& ap, const MatInfo& mt, const ApplyBlock& k,
                                                  int lane, const uint32_t (&o)[16], const float (&pv)[32]) {
  const int64_t cols = mt.cols;
  const int64_t i0 = static_cast<int64_t>(k.r0) * cols + k.c0 + lane;
  float* dst = ap.params + mt.off + i0;
  __nv_bfloat16* dst16 = ap.params_bf16 ? reinterpret_cast<__nv_bfloat16*>(ap.params_bf16) + mt.off + i0 : nullptr;
  const float coef = ap.lr * mt.scale;
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    if (j < k.nr && lane < k.nc) {
      const uint16_t bits = static_cast<uint16_t>((j & 1) ? (o[j >> 1] >> 16) : (o[j >> 1] & 0xffffu));
      const float ov = FP16 ? __half2float(__ushort_as_half(bits)) : __bfloat162float(__ushort_as_bfloat16(bits));
      const float np = fmaf(-coef, ov, pv[j] * ap.decay);
      dst[j * cols] = np;
      if (dst16) dst16[j * cols] = __float2bfloat16_rn(np);
    }
  }
}

}  // namespace
}  // namespace nsm
