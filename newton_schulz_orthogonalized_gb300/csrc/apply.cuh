// The step's decay-and-update applied from a GEMM epilogue, shared by the grouped engine
// and the small-matrix kernel.  The update rule is the one of "DeepSpeed 集成 Muon 优化器实战"
// §核心算子: p <- p (1 - lr wd) - lr sqrt(max(1, rows/cols)) O, both terms on the old p.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
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
