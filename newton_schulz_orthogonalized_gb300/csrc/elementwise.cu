// Memory-bound kernels of the Muon step and the fused AdamW step.
//
//   k_momentum_class  M <- mu M + G and U = G + mu M (Nesterov) or M, in one pass: M
//                     written back, U 2^k (k from the matrix's exponent hint) moved from
//                     the natural row-major layout into the matrix's slot (transposed
//                     when rows > cols) and rounded once to bf16 or fp16; for each warp of
//                     each tile the sum of U^2 and the largest |U|, in fp32 (fixed order)
//   k_grad_norm       per-chunk sums of G^2 and largest |G| (the orthogonalisation)
//   k_scale_finalize  s_i = 1 / (sqrt(sum of matrix i's partial sums) + eps), fixed order;
//                     the exponent k_i that puts max|U| 2^k in [2^11, 2^12); the input
//                     factor s_i 2^-k_i of the chain's products that read X
//   k_to_class        U 2^k (U recomputed in fp32 from G and the updated M, or U = G) into
//                     the slot: the orthogonalisation's layout pass, and the step's second
//                     pass over the matrices whose hint was out of range
//   k_from_class      APPLY: p <- p (1 - lr wd) - lr sqrt(max(1, rows/cols)) O, O read
//                     back from the slot (transposed back when rows > cols), with the
//                     bf16 copy of p when asked; otherwise O copied to a natural bf16
//                     layout (the export of muon_orthogonalize)
//   k_adamw           decoupled-weight-decay Adam on a flat group
//
// The normalised input X = s U is stored as U 2^k: a power of two commutes with the
// rounding wherever U 2^k is a normal value of the format, so the stored X is s times U
// rounded to the format's significant bits, whichever k was used, and s 2^-k enters the
// products that read it in fp32.  A step knows each matrix's norm only after its pass
// over U, so it stores U with the exponent the previous step chose (kept in the
// workspace) and stores it again, in a second pass, only where that exponent put max|U|
// 2^k outside [2^4, 2^15).
//
// The layout kernels work in units of 64 x 64 natural tiles.  A tall matrix's tile is
// transposed through shared memory; a direct matrix whose slot stride equals its width
// has the same layout in both places, so its k-th unit is simply its k-th run of 4096
// consecutive elements.
//
// Sources ("DeepSpeed 集成 Muon 优化器实战" §什么是 Muon 优化器？, §核心算子,
// §混合优化器的参数组构造).  Every reduction runs in a fixed order, so results are
// bit-identical from run to run.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "launch.cuh"
#include "nsm_internal.h"

namespace nsm {
namespace {

constexpr int kThreads = 256;
constexpr int kUFromGrad = 0;   // U = G (orthogonalisation only)
constexpr int kUMomentum = 1;   // U = M (momentum already updated)
constexpr int kUNesterov = 2;   // U = G + mu M

__device__ __forceinline__ int find_by_chunk(const MatInfo* __restrict__ mats, int nmats, int c) {
  int lo = 0, hi = nmats - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mats[mid].chunk_begin <= c) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ int find_by_tile(const MatInfo* __restrict__ mats, int nmats,
                                            int64_t t) {
  int lo = 0, hi = nmats - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (mats[mid].tile_begin <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4& raw, float (&f)[8]) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 t = __bfloat1622float2(h[j]);
    f[2 * j] = t.x;
    f[2 * j + 1] = t.y;
  }
}

__device__ __forceinline__ uint4 pack_bf16x8(const float (&f)[8]) {
  uint4 raw;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
  for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(f[2 * j], f[2 * j + 1]);
  return raw;
}

__device__ __forceinline__ uint4 pack_f16x8(const float (&f)[8]) {
  uint4 raw;
  __half2* h = reinterpret_cast<__half2*>(&raw);
#pragma unroll
  for (int j = 0; j < 4; ++j) h[j] = __floats2half2_rn(f[2 * j], f[2 * j + 1]);
  return raw;
}

__device__ __forceinline__ void unpack_f16x8(const uint4& raw, float (&f)[8]) {
  const __half2* h = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float2 t = __half22float2(h[j]);
    f[2 * j] = t.x;
    f[2 * j + 1] = t.y;
  }
}

template <bool FP16>
__device__ __forceinline__ float load_half(const void* base, int64_t i) {
  if (FP16) return __half2float(reinterpret_cast<const __half*>(base)[i]);
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
}

template <bool FP16>
__device__ __forceinline__ void store_half(void* base, int64_t i, float v) {
  if (FP16) reinterpret_cast<__half*>(base)[i] = __float2half_rn(v);
  else reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(v);
}

template <bool FP16>
__device__ __forceinline__ void load8(const void* base, int64_t i, float (&f)[8]) {
  const uint4 raw = *reinterpret_cast<const uint4*>(
      reinterpret_cast<const uint16_t*>(base) + i);
  if (FP16) unpack_f16x8(raw, f); else unpack_bf16x8(raw, f);
}

template <bool FP16>
__device__ __forceinline__ void store8(void* base, int64_t i, const float (&f)[8]) {
  *reinterpret_cast<uint4*>(reinterpret_cast<uint16_t*>(base) + i) =
      FP16 ? pack_f16x8(f) : pack_bf16x8(f);
}

// Sum and largest value over the block, in a fixed order; valid in thread 0.  One barrier:
// a caller that reduces again alternates between two scratch buffers.
__device__ __forceinline__ void block_sum_max(float& sum, float& mx, float (*scratch)[kThreads / 32]) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sum += __shfl_xor_sync(0xffffffffu, sum, o);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  }
  const int warp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    scratch[0][warp] = sum;
    scratch[1][warp] = mx;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    sum = 0.f;
    mx = 0.f;
    for (int w = 0; w < kThreads / 32; ++w) {
      sum += scratch[0][w];
      mx = fmaxf(mx, scratch[1][w]);
    }
  }
}

// 2^k for k in [-126, 127] (built from its bits: exact)
__device__ __forceinline__ float pow2f(int k) { return __int_as_float((k + 127) << 23); }

// ---------------------------------------------------------------- bounds checks

// Tests of the checked build (bounds_ok; compiled out otherwise).  natural_run: w
// elements from element i of a matrix of len elements in the packed natural layout, whose
// first element is element `base` of the buffer.  slot_run: w elements from (row, col) of
// a matrix's slot (m rows of n elements, row stride ld).  Runs of 8 are 16-byte vectors
// (8 x 16-bit, or 2 x 4 fp32 at the same index) and must start on a multiple of 8
// elements.
__device__ __forceinline__ bool natural_run(int64_t base, int64_t i, int w, int64_t len) {
  return i >= 0 && i + w <= len && (w == 1 || ((base + i) & 7) == 0);
}

__device__ __forceinline__ bool slot_run(const MatInfo& mt, int row, int col, int w) {
  return row >= 0 && row < mt.m && col >= 0 && col + w <= mt.n &&
         (w == 1 || ((mt.slot + static_cast<int64_t>(row) * mt.ld + col) & 7) == 0);
}

// ---------------------------------------------------------------- norms

// Per chunk of kChunk natural elements: sum of G^2 and largest |G|.
__global__ void __launch_bounds__(kThreads)
    k_grad_norm(const __nv_bfloat16* __restrict__ grads, const MatInfo* __restrict__ mats, int nmats,
                int total_chunks, float* __restrict__ partials, int* status) {
  grid_dependency_sync();  // inputs come from the previous kernel of the stream
  release_dependents();
  __shared__ float scratch[2][2][kThreads / 32];
  constexpr int K = NSM_KERNEL_MOMENTUM;
  int rb = 0;
  for (int chunk = blockIdx.x; chunk < total_chunks; chunk += gridDim.x) {
    const MatInfo& mt = mats[find_by_chunk(mats, nmats, chunk)];
    const int64_t len = static_cast<int64_t>(mt.rows) * mt.cols;
    const int64_t start = static_cast<int64_t>(chunk - mt.chunk_begin) * kChunk;
    const int64_t end = min(start + static_cast<int64_t>(kChunk), len);
    const __nv_bfloat16* g = grads + mt.off;
    float acc = 0.f, mx = 0.f;
    const int64_t nvec = (end - start) >> 3;
    for (int64_t v = threadIdx.x; v < nvec; v += kThreads) {
      const int64_t i = start + v * 8;
      if (!bounds_ok(natural_run(mt.off, i, 8, len), status, K, 0, NSM_SITE_NATURAL_LOAD)) continue;
      float gf[8];
      unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(g + i)), gf);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        acc = fmaf(gf[j], gf[j], acc);
        mx = fmaxf(mx, fabsf(gf[j]));
      }
    }
    for (int64_t i = start + nvec * 8 + threadIdx.x; i < end; i += kThreads) {
      if (!bounds_ok(natural_run(mt.off, i, 1, len), status, K, 0, NSM_SITE_NATURAL_LOAD)) continue;
      const float gv = __bfloat162float(g[i]);
      acc = fmaf(gv, gv, acc);
      mx = fmaxf(mx, fabsf(gv));
    }
    block_sum_max(acc, mx, scratch[rb]);
    if (threadIdx.x == 0) {
      partials[chunk] = acc;
      partials[total_chunks + chunk] = mx;
    }
    rb ^= 1;
  }
}

// One block per matrix: sums and maxima of its partials (per unit: one per chunk, or
// kTileParts per tile when by_tile; the maxima nparts units after the sums), then s, the
// exponent and the input factor.
__global__ void __launch_bounds__(kThreads)
    k_scale_finalize(const MatInfo* __restrict__ mats, int nmats, const float* __restrict__ parts,
                     int64_t nparts, int by_tile, int* __restrict__ hints, float* __restrict__ layout_scale,
                     int* __restrict__ redo, float* __restrict__ xs, float* __restrict__ xs_cls, float eps) {
  grid_dependency_sync();  // inputs come from the previous kernel of the stream
  release_dependents();
  __shared__ float scratch[2][2][kThreads / 32];
  int rb = 0;
  for (int i = blockIdx.x; i < nmats; i += gridDim.x) {
    const MatInfo& mt = mats[i];
    const int per = by_tile ? kTileParts : 1;  // partials per unit
    const int64_t begin = (by_tile ? mt.tile_begin : mt.chunk_begin) * per;
    const int64_t count = (by_tile ? static_cast<int64_t>((mt.rows + kTile - 1) / kTile) * ((mt.cols + kTile - 1) / kTile)
                                   : mt.nchunks) * per;
    float sum = 0.f, mx = 0.f;
    for (int64_t c = threadIdx.x; c < count; c += kThreads) {
      sum += parts[begin + c];
      mx = fmaxf(mx, parts[nparts * per + begin + c]);
    }
    block_sum_max(sum, mx, scratch[rb]);
    rb ^= 1;
    if (threadIdx.x != 0) continue;
    const float s = 1.0f / (sqrtf(sum) + eps);
    const InExponent r = in_exponent(mx, hints != nullptr, hints ? hints[i] : 0);
    layout_scale[i] = r.store ? pow2f(r.k) : 0.f;
    if (hints) {
      if (r.store) *redo = 1;
      hints[i] = r.next;
    }
    const float f = s * pow2f(-r.k);
    xs[i] = f;
    xs_cls[mt.cls_pos] = f;
  }
}

// ---------------------------------------------------------------- layout moves

struct TilePos {
  int mi;
  int r0, c0;
};

__device__ __forceinline__ TilePos tile_pos(const MatInfo* __restrict__ mats, int nmats, int64_t t) {
  const int mi = find_by_tile(mats, nmats, t);
  const MatInfo& mt = mats[mi];
  const int64_t local = t - mt.tile_begin;
  const int tiles_c = (mt.cols + kTile - 1) / kTile;
  const int tr = static_cast<int>(local / tiles_c);
  const int tc = static_cast<int>(local - static_cast<int64_t>(tr) * tiles_c);
  return {mi, tr * kTile, tc * kTile};
}

// U of eight consecutive natural elements: G (no momentum), M (plain momentum, already
// updated) or G + mu M (Nesterov).
template <int MODE>
__device__ __forceinline__ void load_u8(const __nv_bfloat16* g, const float* m, int64_t i, float mu,
                                        float (&u)[8]) {
  unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(g + i)), u);
  if (MODE != kUFromGrad) {
    const float4 m0 = __ldg(reinterpret_cast<const float4*>(m + i));
    const float4 m1 = __ldg(reinterpret_cast<const float4*>(m + i + 4));
    const float mf[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
    for (int q = 0; q < 8; ++q) u[q] = (MODE == kUNesterov) ? fmaf(mu, mf[q], u[q]) : mf[q];
  }
}

template <int MODE>
__device__ __forceinline__ float load_u1(const __nv_bfloat16* g, const float* m, int64_t i, float mu) {
  if (MODE == kUFromGrad) return __bfloat162float(g[i]);
  if (MODE == kUMomentum) return m[i];
  return fmaf(mu, m[i], __bfloat162float(g[i]));
}

// The step's pass over G and M: M <- mu M + G written back in place, U = G + mu M
// (Nesterov) or M stored as U 2^k (k = the matrix's hint) into the slot (row stride ld),
// transposed when rows > cols, rounded once to bf16/fp16; for each warp w of tile t the
// sum of U^2 and the largest |U| over its elements (tparts[t kTileParts + w], and
// kTileParts total_tiles entries later).
template <bool TO_FP16, bool NESTEROV>
__global__ void __launch_bounds__(kThreads)
    k_momentum_class(const __nv_bfloat16* __restrict__ grads, float* __restrict__ mom, float mu,
                     void* __restrict__ dst, const MatInfo* __restrict__ mats, int nmats,
                     int64_t total_tiles, const int* __restrict__ hints, float* __restrict__ tparts,
                     int* __restrict__ redo, int* status) {
  grid_dependency_sync();  // inputs come from the previous kernel of the stream
  release_dependents();
  __shared__ float tile[kTile][kTile + 1];
  static_assert(kTileParts == kThreads / 32, "one partial sum and maximum per warp and tile");
  constexpr int K = NSM_KERNEL_MOMENTUM;
  if (blockIdx.x == 0 && threadIdx.x == 0) *redo = 0;  // the finalize kernel sets it
  for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x) {
    const TilePos tp = tile_pos(mats, nmats, t);
    const MatInfo& mt = mats[tp.mi];
    const __nv_bfloat16* g = grads + mt.off;
    float* m = mom + mt.off;
    const int64_t d0 = mt.slot;
    const float sc = pow2f(in_clamp_exp(hints[tp.mi]));
    const int rows = mt.rows, cols = mt.cols, ld = mt.ld;
    const int64_t len = static_cast<int64_t>(rows) * cols;
    float acc = 0.f, mx = 0.f;
    // G read, M read and written at the eight natural elements from i; U into u
    auto step8 = [&](int64_t i, float (&u)[8]) {
      float gf[8];
      unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(g + i)), gf);
      float4* mp = reinterpret_cast<float4*>(m + i);
      const float4 m0 = mp[0], m1 = mp[1];
      float mf[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float mn = fmaf(mu, mf[j], gf[j]);
        mf[j] = mn;
        u[j] = NESTEROV ? fmaf(mu, mn, gf[j]) : mn;
        acc = fmaf(u[j], u[j], acc);
        mx = fmaxf(mx, fabsf(u[j]));
      }
      mp[0] = make_float4(mf[0], mf[1], mf[2], mf[3]);
      mp[1] = make_float4(mf[4], mf[5], mf[6], mf[7]);
    };
    auto step1 = [&](int64_t i) {
      const float gv = __bfloat162float(g[i]);
      const float mn = fmaf(mu, m[i], gv);
      m[i] = mn;
      const float uv = NESTEROV ? fmaf(mu, mn, gv) : mn;
      acc = fmaf(uv, uv, acc);
      mx = fmaxf(mx, fabsf(uv));
      return uv;
    };
    if (!mt.transposed) {
      if ((mt.flags & kMatVec) && ld == cols) {
        // slot and natural layouts coincide: the matrix's k-th tile is its k-th run of
        // kTile^2 consecutive elements, streamed contiguously
        const int64_t base = (t - mt.tile_begin) * (kTile * kTile);
        for (int j = threadIdx.x; j < kTile * kTile / 8; j += kThreads) {
          const int64_t i = base + static_cast<int64_t>(j) * 8;
          if (i < len) {
            if (!bounds_ok(natural_run(mt.off, i, 8, len), status, K, 0, NSM_SITE_NATURAL_LOAD)) continue;
            float u[8];
            step8(i, u);
#pragma unroll
            for (int q = 0; q < 8; ++q) u[q] *= sc;
            if (!bounds_ok(slot_run(mt, static_cast<int>(i / ld), static_cast<int>(i % ld), 8), status, K, 0,
                           NSM_SITE_SLOT_STORE)) continue;
            store8<TO_FP16>(dst, d0 + i, u);
          }
        }
      } else if (mt.flags & kMatVec) {
        for (int j = threadIdx.x; j < kTile * kTile / 8; j += kThreads) {
          const int r = tp.r0 + (j >> 3), c = tp.c0 + (j & 7) * 8;
          if (r < rows && c < cols) {
            const int64_t i = static_cast<int64_t>(r) * cols + c;
            if (!bounds_ok(natural_run(mt.off, i, 8, len), status, K, 0, NSM_SITE_NATURAL_LOAD)) continue;
            float u[8];
            step8(i, u);
#pragma unroll
            for (int q = 0; q < 8; ++q) u[q] *= sc;
            if (!bounds_ok(slot_run(mt, r, c, 8), status, K, 0, NSM_SITE_SLOT_STORE)) continue;
            store8<TO_FP16>(dst, d0 + static_cast<int64_t>(r) * ld + c, u);
          }
        }
      } else {
        for (int j = threadIdx.x; j < kTile * kTile; j += kThreads) {
          const int r = tp.r0 + (j >> 6), c = tp.c0 + (j & 63);
          if (r < rows && c < cols) {
            const int64_t i = static_cast<int64_t>(r) * cols + c;
            if (!bounds_ok(natural_run(mt.off, i, 1, len), status, K, 0, NSM_SITE_NATURAL_LOAD)) continue;
            const float v = step1(i) * sc;
            if (!bounds_ok(slot_run(mt, r, c, 1), status, K, 0, NSM_SITE_SLOT_STORE)) continue;
            store_half<TO_FP16>(dst, d0 + static_cast<int64_t>(r) * ld + c, v);
          }
        }
      }
    } else {
      // slot row = natural column c, slot column = natural row r
      if (mt.flags & kMatVec) {
        for (int j = threadIdx.x; j < kTile * kTile / 8; j += kThreads) {
          const int rr = j >> 3, cc = (j & 7) * 8;
          const int r = tp.r0 + rr, c = tp.c0 + cc;
          float u[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (r < rows && c < cols &&
              bounds_ok(natural_run(mt.off, static_cast<int64_t>(r) * cols + c, 8, len), status, K, 0,
                        NSM_SITE_NATURAL_LOAD)) {
            step8(static_cast<int64_t>(r) * cols + c, u);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) tile[rr][cc + q] = u[q];
        }
        __syncthreads();
        for (int j = threadIdx.x; j < kTile * kTile / 8; j += kThreads) {
          const int cr = j >> 3, rc = (j & 7) * 8;  // slot row c0+cr, slot cols r0+rc..+7
          const int c = tp.c0 + cr, r = tp.r0 + rc;
          if (c < cols && r < rows && bounds_ok(slot_run(mt, c, r, 8), status, K, 0, NSM_SITE_SLOT_STORE)) {
            float f[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] = tile[rc + q][cr] * sc;
            store8<TO_FP16>(dst, d0 + static_cast<int64_t>(c) * ld + r, f);
          }
        }
      } else {
        for (int j = threadIdx.x; j < kTile * kTile; j += kThreads) {
          const int rr = j >> 6, cc = j & 63;
          const int r = tp.r0 + rr, c = tp.c0 + cc;
          const bool in = r < rows && c < cols &&
                          bounds_ok(natural_run(mt.off, static_cast<int64_t>(r) * cols + c, 1, len), status, K, 0,
                                    NSM_SITE_NATURAL_LOAD);
          tile[rr][cc] = in ? step1(static_cast<int64_t>(r) * cols + c) : 0.f;
        }
        __syncthreads();
        for (int j = threadIdx.x; j < kTile * kTile; j += kThreads) {
          const int cr = j >> 6, rc = j & 63;
          const int c = tp.c0 + cr, r = tp.r0 + rc;
          if (c < cols && r < rows && bounds_ok(slot_run(mt, c, r, 1), status, K, 0, NSM_SITE_SLOT_STORE)) {
            store_half<TO_FP16>(dst, d0 + static_cast<int64_t>(c) * ld + r, tile[rc][cr] * sc);
          }
        }
      }
      __syncthreads();
    }
    // each warp's sum and maximum over its elements of the tile, in a fixed order
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      acc += __shfl_xor_sync(0xffffffffu, acc, o);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    if ((threadIdx.x & 31) == 0) {
      const int part = static_cast<int>(threadIdx.x >> 5);
      tparts[t * kTileParts + part] = acc;
      tparts[(total_tiles + t) * kTileParts + part] = mx;
    }
  }
}

// X = U 2^k (scales[i] = 2^k) moved from the natural row-major layout (row stride cols)
// into the matrix's slot (row stride ld), transposed when rows > cols, rounded once to
// bf16/fp16.  redo != NULL (the step's second pass): nothing is done when *redo is 0, and
// matrices whose scale is 0 keep what their slot holds.
template <bool TO_FP16, int MODE>
__global__ void __launch_bounds__(kThreads)
    k_to_class(const __nv_bfloat16* __restrict__ grads, const float* __restrict__ mom, float mu,
               void* __restrict__ dst, const MatInfo* __restrict__ mats, int nmats,
               int64_t total_tiles, const float* __restrict__ scales, const int* __restrict__ redo,
               int* status) {
  grid_dependency_sync();  // inputs come from the previous kernel of the stream
  release_dependents();
  __shared__ float tile[kTile][kTile + 1];
  if (redo && *redo == 0) return;  // the step's second pass: nothing to store again
  for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x) {
    const TilePos tp = tile_pos(mats, nmats, t);
    const MatInfo& mt = mats[tp.mi];
    const float sc = scales[tp.mi];
    if (redo && sc == 0.f) {
      // on to this block's first tile of a later matrix (the same for all threads)
      const int64_t end = tp.mi + 1 < nmats ? mats[tp.mi + 1].tile_begin : total_tiles;
      t += (end - 1 - t) / gridDim.x * gridDim.x;
      continue;
    }
    const __nv_bfloat16* g = grads + mt.off;
    const float* m = (MODE == kUFromGrad) ? nullptr : mom + mt.off;
    const int64_t d0 = mt.slot;
    const int rows = mt.rows, cols = mt.cols, ld = mt.ld;
    const int64_t len = static_cast<int64_t>(rows) * cols;
    constexpr int K = NSM_KERNEL_TO_CLASS;
    if (!mt.transposed) {
      if ((mt.flags & kMatVec) && ld == cols) {
        // slot and natural layouts coincide: the matrix's k-th tile is its k-th run of
        // kTile^2 consecutive elements, streamed contiguously
        const int64_t base = (t - mt.tile_begin) * (kTile * kTile);
        for (int j = threadIdx.x; j < kTile * kTile / 8; j += kThreads) {
          const int64_t i = base + static_cast<int64_t>(j) * 8;
          if (i < len) {
            float f[8];
            if (!bounds_ok(natural_run(mt.off, i, 8, len), status, K, 0, NSM_SITE_NATURAL_LOAD)) continue;
            load_u8<MODE>(g, m, i, mu, f);
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] *= sc;
            if (!bounds_ok(slot_run(mt, static_cast<int>(i / ld), static_cast<int>(i % ld), 8), status, K, 0,
                           NSM_SITE_SLOT_STORE)) continue;
            store8<TO_FP16>(dst, d0 + i, f);
          }
        }
      } else if (mt.flags & kMatVec) {
        for (int j = threadIdx.x; j < kTile * kTile / 8; j += kThreads) {
          const int r = tp.r0 + (j >> 3), c = tp.c0 + (j & 7) * 8;
          if (r < rows && c < cols) {
            float f[8];
            const int64_t i = static_cast<int64_t>(r) * cols + c;
            if (!bounds_ok(natural_run(mt.off, i, 8, len), status, K, 0, NSM_SITE_NATURAL_LOAD)) continue;
            load_u8<MODE>(g, m, i, mu, f);
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] *= sc;
            if (!bounds_ok(slot_run(mt, r, c, 8), status, K, 0, NSM_SITE_SLOT_STORE)) continue;
            store8<TO_FP16>(dst, d0 + static_cast<int64_t>(r) * ld + c, f);
          }
        }
      } else {
        for (int j = threadIdx.x; j < kTile * kTile; j += kThreads) {
          const int r = tp.r0 + (j >> 6), c = tp.c0 + (j & 63);
          if (r < rows && c < cols) {
            const int64_t i = static_cast<int64_t>(r) * cols + c;
            if (!bounds_ok(natural_run(mt.off, i, 1, len), status, K, 0, NSM_SITE_NATURAL_LOAD)) continue;
            const float v = load_u1<MODE>(g, m, i, mu) * sc;
            if (!bounds_ok(slot_run(mt, r, c, 1), status, K, 0, NSM_SITE_SLOT_STORE)) continue;
            store_half<TO_FP16>(dst, d0 + static_cast<int64_t>(r) * ld + c, v);
          }
        }
      }
    } else {
      // slot row = natural column c, slot column = natural row r
      if (mt.flags & kMatVec) {
        for (int j = threadIdx.x; j < kTile * kTile / 8; j += kThreads) {
          const int rr = j >> 3, cc = (j & 7) * 8;
          const int r = tp.r0 + rr, c = tp.c0 + cc;
          float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (r < rows && c < cols &&
              bounds_ok(natural_run(mt.off, static_cast<int64_t>(r) * cols + c, 8, len), status, K, 0,
                        NSM_SITE_NATURAL_LOAD)) {
            load_u8<MODE>(g, m, static_cast<int64_t>(r) * cols + c, mu, f);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) tile[rr][cc + q] = f[q];
        }
        __syncthreads();
        for (int j = threadIdx.x; j < kTile * kTile / 8; j += kThreads) {
          const int cr = j >> 3, rc = (j & 7) * 8;  // slot row c0+cr, slot cols r0+rc..+7
          const int c = tp.c0 + cr, r = tp.r0 + rc;
          if (c < cols && r < rows && bounds_ok(slot_run(mt, c, r, 8), status, K, 0, NSM_SITE_SLOT_STORE)) {
            float f[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] = tile[rc + q][cr] * sc;
            store8<TO_FP16>(dst, d0 + static_cast<int64_t>(c) * ld + r, f);
          }
        }
      } else {
        for (int j = threadIdx.x; j < kTile * kTile; j += kThreads) {
          const int rr = j >> 6, cc = j & 63;
          const int r = tp.r0 + rr, c = tp.c0 + cc;
          const bool in = r < rows && c < cols &&
                          bounds_ok(natural_run(mt.off, static_cast<int64_t>(r) * cols + c, 1, len), status, K, 0,
                                    NSM_SITE_NATURAL_LOAD);
          tile[rr][cc] = in ? load_u1<MODE>(g, m, static_cast<int64_t>(r) * cols + c, mu) : 0.f;
        }
        __syncthreads();
        for (int j = threadIdx.x; j < kTile * kTile; j += kThreads) {
          const int cr = j >> 6, rc = j & 63;
          const int c = tp.c0 + cr, r = tp.r0 + rc;
          if (c < cols && r < rows && bounds_ok(slot_run(mt, c, r, 1), status, K, 0, NSM_SITE_SLOT_STORE)) {
            store_half<TO_FP16>(dst, d0 + static_cast<int64_t>(c) * ld + r, tile[rc][cr] * sc);
          }
        }
      }
      __syncthreads();
    }
  }
}

// Slot O -> natural layout, O being the stored values times oscale[i] (NULL: 1).  APPLY:
// p <- p*decay - lr*scale*O, and out = bf16(p) when out is not NULL (the parameters' bf16
// copy).  Otherwise out = bf16(O).
template <bool O_FP16, bool APPLY>
__global__ void __launch_bounds__(kThreads)
    k_from_class(const void* __restrict__ o, const float* __restrict__ oscale, float* __restrict__ params,
                 __nv_bfloat16* __restrict__ out, const MatInfo* __restrict__ mats, int nmats,
                 int64_t total_tiles, float lr, float decay, int* status) {
  grid_dependency_sync();  // inputs come from the previous kernel of the stream
  release_dependents();
  __shared__ float tile[kTile][kTile + 1];
  constexpr int K = NSM_KERNEL_FROM_CLASS;
  // p is read and written (and its bf16 copy written) at the same elements; the export
  // only writes its bf16 output there
  constexpr int kNatural = APPLY ? NSM_SITE_NATURAL_LOAD : NSM_SITE_NATURAL_STORE;
  for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x) {
    const TilePos tp = tile_pos(mats, nmats, t);
    const MatInfo& mt = mats[tp.mi];
    const int rows = mt.rows, cols = mt.cols, ld = mt.ld;
    const int64_t len = static_cast<int64_t>(rows) * cols;
    const int64_t s0 = mt.slot;
    const float os = oscale ? oscale[tp.mi] : 1.f;  // times 1 leaves every value as it is
    const float coef = lr * mt.scale * os;
    float* p = APPLY ? params + mt.off : nullptr;
    __nv_bfloat16* ob = out ? out + mt.off : nullptr;
    if (mt.transposed) {
      // tile[rr][cc] = O^T[r0+rr][c0+cc] = slot[c0+cc][r0+rr]
      if (mt.flags & kMatVec) {
        for (int j = threadIdx.x; j < kTile * kTile / 8; j += kThreads) {
          const int cc = j >> 3, rr = (j & 7) * 8;
          const int c = tp.c0 + cc, r = tp.r0 + rr;
          float f[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          if (c < cols && r < rows && bounds_ok(slot_run(mt, c, r, 8), status, K, 0, NSM_SITE_SLOT_LOAD)) {
            load8<O_FP16>(o, s0 + static_cast<int64_t>(c) * ld + r, f);
          }
#pragma unroll
          for (int q = 0; q < 8; ++q) tile[rr + q][cc] = f[q];
        }
      } else {
        for (int j = threadIdx.x; j < kTile * kTile; j += kThreads) {
          const int cc = j >> 6, rr = j & 63;
          const int c = tp.c0 + cc, r = tp.r0 + rr;
          const bool in = c < cols && r < rows && bounds_ok(slot_run(mt, c, r, 1), status, K, 0, NSM_SITE_SLOT_LOAD);
          tile[rr][cc] = in ? load_half<O_FP16>(o, s0 + static_cast<int64_t>(c) * ld + r) : 0.f;
        }
      }
      __syncthreads();
    }
    if ((mt.flags & kMatVec) && !mt.transposed && ld == cols) {
      // slot and natural layouts coincide: the k-th tile is the k-th run of kTile^2
      // consecutive elements
      const int64_t base = (t - mt.tile_begin) * (kTile * kTile);
      for (int j = threadIdx.x; j < kTile * kTile / 8; j += kThreads) {
        const int64_t i = base + static_cast<int64_t>(j) * 8;
        if (i < len) {
          float f[8];
          if (!bounds_ok(slot_run(mt, static_cast<int>(i / ld), static_cast<int>(i % ld), 8), status, K, 0,
                         NSM_SITE_SLOT_LOAD)) continue;
          if (!bounds_ok(natural_run(mt.off, i, 8, len), status, K, 0, kNatural)) continue;
          load8<O_FP16>(o, s0 + i, f);
          if (APPLY) {
            float4* pp = reinterpret_cast<float4*>(p + i);
            float4 a = pp[0], b = pp[1];
            a.x = fmaf(-coef, f[0], a.x * decay);
            a.y = fmaf(-coef, f[1], a.y * decay);
            a.z = fmaf(-coef, f[2], a.z * decay);
            a.w = fmaf(-coef, f[3], a.w * decay);
            b.x = fmaf(-coef, f[4], b.x * decay);
            b.y = fmaf(-coef, f[5], b.y * decay);
            b.z = fmaf(-coef, f[6], b.z * decay);
            b.w = fmaf(-coef, f[7], b.w * decay);
            pp[0] = a;
            pp[1] = b;
            if (ob) {
              const float np[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
              *reinterpret_cast<uint4*>(ob + i) = pack_bf16x8(np);
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] *= os;
            *reinterpret_cast<uint4*>(ob + i) = pack_bf16x8(f);
          }
        }
      }
    } else if (mt.flags & kMatVec) {
      for (int j = threadIdx.x; j < kTile * kTile / 8; j += kThreads) {
        const int rr = j >> 3, cc = (j & 7) * 8;
        const int r = tp.r0 + rr, c = tp.c0 + cc;
        if (r < rows && c < cols) {
          float f[8];
          const int64_t i = static_cast<int64_t>(r) * cols + c;
          if (!bounds_ok(natural_run(mt.off, i, 8, len), status, K, 0, kNatural)) continue;
          if (mt.transposed) {
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] = tile[rr][cc + q];
          } else {
            if (!bounds_ok(slot_run(mt, r, c, 8), status, K, 0, NSM_SITE_SLOT_LOAD)) continue;
            load8<O_FP16>(o, s0 + static_cast<int64_t>(r) * ld + c, f);
          }
          if (APPLY) {
            float4* pp = reinterpret_cast<float4*>(p + i);
            float4 a = pp[0], b = pp[1];
            a.x = fmaf(-coef, f[0], a.x * decay);
            a.y = fmaf(-coef, f[1], a.y * decay);
            a.z = fmaf(-coef, f[2], a.z * decay);
            a.w = fmaf(-coef, f[3], a.w * decay);
            b.x = fmaf(-coef, f[4], b.x * decay);
            b.y = fmaf(-coef, f[5], b.y * decay);
            b.z = fmaf(-coef, f[6], b.z * decay);
            b.w = fmaf(-coef, f[7], b.w * decay);
            pp[0] = a;
            pp[1] = b;
            if (ob) {
              const float np[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
              *reinterpret_cast<uint4*>(ob + i) = pack_bf16x8(np);
            }
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) f[q] *= os;
            *reinterpret_cast<uint4*>(ob + i) = pack_bf16x8(f);
          }
        }
      }
    } else {
      for (int j = threadIdx.x; j < kTile * kTile; j += kThreads) {
        const int rr = j >> 6, cc = j & 63;
        const int r = tp.r0 + rr, c = tp.c0 + cc;
        if (r < rows && c < cols) {
          const int64_t i = static_cast<int64_t>(r) * cols + c;
          if (!bounds_ok(natural_run(mt.off, i, 1, len), status, K, 0, kNatural)) continue;
          if (!mt.transposed && !bounds_ok(slot_run(mt, r, c, 1), status, K, 0, NSM_SITE_SLOT_LOAD)) continue;
          const float ov = mt.transposed ? tile[rr][cc]
                                         : load_half<O_FP16>(o, s0 + static_cast<int64_t>(r) * ld + c);
          if (APPLY) {
            const float np = fmaf(-coef, ov, p[i] * decay);
            p[i] = np;
            if (ob) ob[i] = __float2bfloat16_rn(np);
          } else {
            ob[i] = __float2bfloat16_rn(ov * os);
          }
        }
      }
    }
    if (mt.transposed) __syncthreads();
  }
}

// ---------------------------------------------------------------- AdamW

__device__ __forceinline__ void adamw_elem(float g, float& p, float& m, float& v, float b1,
                                           float b2, float eps, float decay, float step_size,
                                           float bc2) {
  m = fmaf(b1, m, (1.0f - b1) * g);
  v = fmaf(b2, v, (1.0f - b2) * g * g);
  const float denom = sqrtf(v / bc2) + eps;
  p = p * decay - step_size * (m / denom);
}

__global__ void __launch_bounds__(kThreads)
    k_adamw(const __nv_bfloat16* __restrict__ grads, float* __restrict__ params,
            float* __restrict__ mom1, float* __restrict__ mom2, int64_t numel, float b1,
            float b2, float eps, float decay, float step_size, float bc2, int* status) {
  grid_dependency_sync();  // inputs come from the previous kernel of the stream
  release_dependents();
  const int64_t nvec = numel >> 3;
  const int64_t stride = static_cast<int64_t>(gridDim.x) * kThreads;
  // two 8-element groups per iteration, every load issued before the first store
  for (int64_t v = blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; v < nvec; v += 2 * stride) {
    // g, p, m and v are read and written at the same 8 elements of the group
    if (!bounds_ok(natural_run(0, v * 8, 8, numel), status, NSM_KERNEL_ADAMW, 0, NSM_SITE_FLAT)) continue;
    const bool two = v + stride < nvec &&
                     bounds_ok(natural_run(0, (v + stride) * 8, 8, numel), status, NSM_KERNEL_ADAMW, 0, NSM_SITE_FLAT);
    float g[2][8];
    float4 p[2][2], m[2][2], w[2][2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u == 1 && !two) break;
      const int64_t i = (v + u * stride) * 8;
      unpack_bf16x8(__ldg(reinterpret_cast<const uint4*>(grads + i)), g[u]);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        p[u][h] = reinterpret_cast<const float4*>(params + i)[h];
        m[u][h] = reinterpret_cast<const float4*>(mom1 + i)[h];
        w[u][h] = reinterpret_cast<const float4*>(mom2 + i)[h];
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u == 1 && !two) break;
      const int64_t i = (v + u * stride) * 8;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        adamw_elem(g[u][4 * h + 0], p[u][h].x, m[u][h].x, w[u][h].x, b1, b2, eps, decay, step_size, bc2);
        adamw_elem(g[u][4 * h + 1], p[u][h].y, m[u][h].y, w[u][h].y, b1, b2, eps, decay, step_size, bc2);
        adamw_elem(g[u][4 * h + 2], p[u][h].z, m[u][h].z, w[u][h].z, b1, b2, eps, decay, step_size, bc2);
        adamw_elem(g[u][4 * h + 3], p[u][h].w, m[u][h].w, w[u][h].w, b1, b2, eps, decay, step_size, bc2);
        reinterpret_cast<float4*>(params + i)[h] = p[u][h];
        reinterpret_cast<float4*>(mom1 + i)[h] = m[u][h];
        reinterpret_cast<float4*>(mom2 + i)[h] = w[u][h];
      }
    }
  }
  for (int64_t i = nvec * 8 + blockIdx.x * static_cast<int64_t>(kThreads) + threadIdx.x; i < numel; i += stride) {
    if (!bounds_ok(natural_run(0, i, 1, numel), status, NSM_KERNEL_ADAMW, 0, NSM_SITE_FLAT)) continue;
    float p = params[i], m = mom1[i], w = mom2[i];
    adamw_elem(__bfloat162float(grads[i]), p, m, w, b1, b2, eps, decay, step_size, bc2);
    params[i] = p;
    mom1[i] = m;
    mom2[i] = w;
  }
}

// ---------------------------------------------------------------- host -> device copy

// Copy from page-locked host memory (through its device mapping) into device memory with
// SM loads: 16-byte units, four in flight per thread, then the trailing bytes.
__global__ void __launch_bounds__(kThreads)
    k_copy_h2d(const uint4* __restrict__ src, uint4* __restrict__ dst, size_t units,
               const uint8_t* __restrict__ src_tail, uint8_t* __restrict__ dst_tail, int tail) {
  const size_t stride = static_cast<size_t>(gridDim.x) * kThreads;
  size_t i = blockIdx.x * static_cast<size_t>(kThreads) + threadIdx.x;
  for (; i + 3 * stride < units; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < units; i += stride) dst[i] = src[i];
  if (blockIdx.x == 0 && static_cast<int>(threadIdx.x) < tail) dst_tail[threadIdx.x] = src_tail[threadIdx.x];
}

int g_num_sms_cache[64] = {0};

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (dev >= 0 && dev < 64 && g_num_sms_cache[dev] > 0) return g_num_sms_cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
  if (dev >= 0 && dev < 64) g_num_sms_cache[dev] = n;
  return n;
}

int grid_for(int64_t items, int per_sm) {
  const int64_t cap = static_cast<int64_t>(num_sms()) * per_sm;
  const int64_t g = items < cap ? items : cap;
  return static_cast<int>(g < 1 ? 1 : g);
}

}  // namespace

cudaError_t launch_grad_norm(const void* grads, const MatInfo* mats, int nmats, int total_chunks,
                             float* partials, cudaStream_t stream) {
  const int grid = grid_for(total_chunks, 8);
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  const auto* g = reinterpret_cast<const __nv_bfloat16*>(grads);
  if (const cudaError_t e_launch = launch_pdl(k_grad_norm, dim3(grid), dim3(kThreads), 0, stream, g, mats, nmats,
                                              total_chunks, partials, status)) return e_launch;
  return cudaGetLastError();
}

cudaError_t launch_momentum_class(const void* grads, float* momentum, int nesterov, float mu, void* dst,
                                  int to_fp16, const MatInfo* mats, int nmats, int64_t total_tiles,
                                  const int* hints, float* tparts, int* redo, cudaStream_t stream) {
  const int grid = grid_for(total_tiles, 8);
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  const auto* g = reinterpret_cast<const __nv_bfloat16*>(grads);
  cudaError_t e;
  if (to_fp16) {
    e = nesterov ? launch_pdl(k_momentum_class<true, true>, dim3(grid), dim3(kThreads), 0, stream, g, momentum, mu,
                              dst, mats, nmats, total_tiles, hints, tparts, redo, status)
                 : launch_pdl(k_momentum_class<true, false>, dim3(grid), dim3(kThreads), 0, stream, g, momentum, mu,
                              dst, mats, nmats, total_tiles, hints, tparts, redo, status);
  } else {
    e = nesterov ? launch_pdl(k_momentum_class<false, true>, dim3(grid), dim3(kThreads), 0, stream, g, momentum, mu,
                              dst, mats, nmats, total_tiles, hints, tparts, redo, status)
                 : launch_pdl(k_momentum_class<false, false>, dim3(grid), dim3(kThreads), 0, stream, g, momentum, mu,
                              dst, mats, nmats, total_tiles, hints, tparts, redo, status);
  }
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_scale_finalize(const MatInfo* mats, int nmats, const float* parts, int64_t nparts,
                                  int by_tile, int* hints, float* layout_scale, int* redo, float* xs,
                                  float* xs_cls, float eps, cudaStream_t stream) {
  const int grid = nmats < 65535 ? nmats : 65535;
  if (const cudaError_t e_launch = launch_pdl(k_scale_finalize, dim3(grid), dim3(kThreads), 0, stream, mats, nmats,
                                              parts, nparts, by_tile, hints, layout_scale, redo, xs, xs_cls, eps))
    return e_launch;
  return cudaGetLastError();
}

template <bool TO_FP16>
static cudaError_t to_class_mode(int mode, int grid, const __nv_bfloat16* g, const float* m, float mu, void* dst,
                          const MatInfo* mats, int nmats, int64_t total_tiles, const float* scales,
                          const int* redo, int* status, cudaStream_t stream) {
  if (mode == kUFromGrad) {
    if (const cudaError_t e_launch = launch_pdl(k_to_class<TO_FP16, kUFromGrad>, dim3(grid), dim3(kThreads), 0, stream, g, m, mu, dst, mats, nmats, total_tiles, scales, redo, status)) return e_launch;
  } else if (mode == kUMomentum) {
    if (const cudaError_t e_launch = launch_pdl(k_to_class<TO_FP16, kUMomentum>, dim3(grid), dim3(kThreads), 0, stream, g, m, mu, dst, mats, nmats, total_tiles, scales, redo, status)) return e_launch;
  } else {
    if (const cudaError_t e_launch = launch_pdl(k_to_class<TO_FP16, kUNesterov>, dim3(grid), dim3(kThreads), 0, stream, g, m, mu, dst, mats, nmats, total_tiles, scales, redo, status)) return e_launch;
  }
  return cudaSuccess;
}

cudaError_t launch_to_class(const void* grads, const float* momentum, int has_momentum, int nesterov, float mu,
                            void* dst, int to_fp16, const MatInfo* mats, int nmats, int64_t total_tiles,
                            const float* scales, const int* redo, cudaStream_t stream) {
  const int grid = grid_for(total_tiles, 8);
  const auto* g = reinterpret_cast<const __nv_bfloat16*>(grads);
  const int mode = !has_momentum ? kUFromGrad : (nesterov ? kUNesterov : kUMomentum);
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  const cudaError_t e = to_fp16 ? to_class_mode<true>(mode, grid, g, momentum, mu, dst, mats, nmats, total_tiles, scales, redo, status, stream)
                                : to_class_mode<false>(mode, grid, g, momentum, mu, dst, mats, nmats, total_tiles, scales, redo, status, stream);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_apply(const void* o, int o_fp16, const float* o_scale, float* params, void* params_bf16,
                         const MatInfo* mats, int nmats, int64_t total_tiles, float lr, float wd,
                         cudaStream_t stream) {
  const int grid = grid_for(total_tiles, 8);
  const float decay = 1.0f - lr * wd;
  auto* pb = reinterpret_cast<__nv_bfloat16*>(params_bf16);
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  if (o_fp16) {
    if (const cudaError_t e_launch = launch_pdl(k_from_class<true, true>, dim3(grid), dim3(kThreads), 0, stream, o, o_scale, params, pb, mats, nmats, total_tiles, lr, decay, status)) return e_launch;
  } else {
    if (const cudaError_t e_launch = launch_pdl(k_from_class<false, true>, dim3(grid), dim3(kThreads), 0, stream, o, o_scale, params, pb, mats, nmats, total_tiles, lr, decay, status)) return e_launch;
  }
  return cudaGetLastError();
}

cudaError_t launch_export(const void* o, int o_fp16, const float* o_scale, void* out, const MatInfo* mats, int nmats,
                          int64_t total_tiles, cudaStream_t stream) {
  const int grid = grid_for(total_tiles, 8);
  auto* ob = reinterpret_cast<__nv_bfloat16*>(out);
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  if (o_fp16) {
    if (const cudaError_t e_launch = launch_pdl(k_from_class<true, false>, dim3(grid), dim3(kThreads), 0, stream, o, o_scale, nullptr, ob, mats, nmats, total_tiles, 0.f, 1.f, status)) return e_launch;
  } else {
    if (const cudaError_t e_launch = launch_pdl(k_from_class<false, false>, dim3(grid), dim3(kThreads), 0, stream, o, o_scale, nullptr, ob, mats, nmats, total_tiles, 0.f, 1.f, status)) return e_launch;
  }
  return cudaGetLastError();
}

cudaError_t launch_copy_h2d(void* dst, const void* src_mapped, size_t bytes, int ctas, cudaStream_t stream) {
  // The copy runs beside the step's kernels, whose persistent GEMM CTAs take nearly all of
  // an SM's shared memory: the copy asks for the same (largest) shared-memory carveout, so
  // that its CTAs do not keep an SM in another configuration.
  const cudaError_t carveout =
      cudaFuncSetAttribute(k_copy_h2d, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
  if (carveout != cudaSuccess) return carveout;
  const size_t units = bytes / 16;
  const int tail = static_cast<int>(bytes % 16);
  const auto* s = static_cast<const uint8_t*>(src_mapped);
  auto* d = static_cast<uint8_t*>(dst);
  k_copy_h2d<<<ctas, kThreads, 0, stream>>>(reinterpret_cast<const uint4*>(s), reinterpret_cast<uint4*>(d), units,
                                            s + units * 16, d + units * 16, tail);
  return cudaGetLastError();
}

cudaError_t launch_adamw(const void* grads, float* params, float* m, float* v, int64_t numel,
                         float lr, float beta1, float beta2, float eps, float wd, float bc1,
                         float bc2, cudaStream_t stream) {
  if (numel <= 0) return cudaSuccess;
  const int64_t items = (numel + 7) / 8;
  const int grid = grid_for((items + kThreads - 1) / kThreads, 8);
  const float decay = 1.0f - lr * wd;
  const float step_size = lr / bc1;
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  if (const cudaError_t e_launch = launch_pdl(k_adamw, dim3(grid), dim3(kThreads), 0, stream, reinterpret_cast<const __nv_bfloat16*>(grads), params, m, v,
                                         numel, beta1, beta2, eps, decay, step_size, bc2, status)) return e_launch;
  return cudaGetLastError();
}

}  // namespace nsm
