// Grouped GEMM engine of the Newton-Schulz chain on the 5th-generation tensor cores.
//
// One persistent launch runs one stage of the chain (for example A = X X^T) for every
// matrix of a packed group.  Matrices of the same working shape form a group whose
// operands sit back to back in the workspace, so one 3D tensor map per buffer covers
// the whole group.  Work units walk the flat tile list with a fixed stride, so every
// output tile is computed by exactly one unit in a fixed order (bit-identical run to run).
//
// Two kernels share the tile decode and the epilogue:
//   k_ns_gemm       one CTA per SM, 128 x 256 tiles (tcgen05.mma.cta_group::1, M = 128).
//   k_ns_gemm_pair  a cluster of two CTAs on two SMs per 256 x 256 tile
//                   (tcgen05.mma.cta_group::2, M = 256): each CTA stages half of A and half
//                   of B, so each SM's shared memory carries two thirds of the operand
//                   traffic of the 1-CTA tile for the same tensor-core work.
// Roles inside a CTA: warp 0 issues TMA loads (128B-swizzled boxes of 64 columns and 64,
// 128 or 256 rows) into a ring of stages, warp 1 issues the MMAs (the leader CTA's, in the
// pair kernel) into two TMEM accumulators of 256 fp32 columns, warps 2-5 drain TMEM with
// tcgen05.ld, apply the fused epilogue  out = alpha*acc + beta*aux + diag*I  and store
// fp16/bf16 32 x 32 blocks through shared memory with TMA stores.  A product that reads
// the chain's input, stored as U 2^k, scales alpha and beta by that problem's s 2^-k
// (squared for X X^T), so that it computes with X = s U.
// A group flagged symmetric computes only the tiles that touch the upper triangle, stores
// the blocks on and above the diagonal and mirrors the upper ones.  In the pair kernel a
// group may instead keep its symmetric m x m buffers as their upper 256 x 256 tiles
// (GemmGroup::lean): the output tiles off the diagonal are stored without a mirror, and a
// K block below an operand's diagonal is loaded from its mirror image as an MN-major
// operand (the A or B major bit of that block's instruction descriptor).
//
// The stages it serves ("DeepSpeed 集成 Muon 优化器实战" §核心算子):
//   standard:  A = X X^T;  B = b A + c A A^T (A symmetric);  X' = a X + B X
//   gram:      R = X X^T;  H = a I + b R + c R R^T;  Q' = H Q^T;  T = H R^T;
//              R' = T H^T;  X = Q X;  O = Q X   (H, Q, R, T symmetric polynomials of R_0)
// B X and Q X read X as a K x N operand with N contiguous ("MN-major").
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "launch.cuh"
#include "nsm_internal.h"
#include "ptx.cuh"

namespace nsm {

__device__ int g_device_status = 0;

int* device_status_ptr() {
  int* p = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_device_status) != cudaSuccess) {
    return nullptr;
  }
  return p;
}

namespace {

constexpr int BN = 256;                   // widest MMA N per tile
constexpr int BK = 64;                    // K per stage: 64 16-bit elements = 128 B rows
constexpr int BOX_BYTES = 64 * 64 * 2;    // one TMA box: 64 rows x 128 B
constexpr int NUM_THREADS = 192;          // 6 warps
constexpr uint32_t TMEM_COLS = 512;       // 2 x 256 fp32 accumulator columns
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // 2 s per wait
constexpr int kPanel = 2;                 // column tiles per raster panel
constexpr int EPI_WARPS = 4;
// Whether the grouped launches may overlap their launch with the previous kernel when
// programmatic dependent launch is on (the NSM_OPT_PDL option).
constexpr bool kOverlapGemmLaunch = true;
constexpr int EPI_STAGE_BYTES = EPI_WARPS * 8192;   // per epilogue warp: 2 slots of 2 x 2 KB staged blocks

// 1-CTA kernel: 128 x 256 tiles, 4 stages of A 16 KB + B 32 KB.
constexpr int S1_STAGES = 4;
constexpr int S1_A_BYTES = 128 * BK * 2;
constexpr int S1_STAGE_BYTES = S1_A_BYTES + BN * BK * 2;

// pair kernel: 256 x 256 tiles, K 128 per stage; each CTA stages A 128 x 128 and half of
// B (128 x 128) as two 128-byte-wide K boxes each: 3 stages of 64 KB.
constexpr int BK2 = 128;
// upper-tile storage (GemmGroup::lean) finds a stage's 256-wide K tile as kb / 2
static_assert(2 * BK2 == BN, "two pair-kernel K stages per 256-wide tile");
constexpr int S2_STAGES = 3;
constexpr int S2_A_BYTES = 128 * BK2 * 2;
constexpr int S2_STAGE_BYTES = S2_A_BYTES + 128 * BK2 * 2;

template <int STAGES>
struct Ctrl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int never;  // stays 0: the flag the teardown waits poll, so they ignore `abort`
};

constexpr size_t S1_SMEM = 1024 + size_t(S1_STAGES) * S1_STAGE_BYTES + EPI_STAGE_BYTES + sizeof(Ctrl<S1_STAGES>);
constexpr size_t S2_SMEM = 1024 + size_t(S2_STAGES) * S2_STAGE_BYTES + EPI_STAGE_BYTES + sizeof(Ctrl<S2_STAGES>);
static_assert(S1_SMEM <= 232448 && S2_SMEM <= 232448, "shared memory per CTA");

struct TileCoord {
  int g, b, m0, n0;
};

// Tile t of the launch: group, matrix within the group, first row and column.  Tiles are
// TILE_M x 256; symmetric groups enumerate their precomputed list, the others the grid in
// panels of kPanel column tiles (rows inside a panel).
template <int TILE_M>
__device__ __forceinline__ TileCoord decode_tile(const GemmGroup* __restrict__ groups, int ng,
                                                 int64_t t) {
  int lo = 0, hi = ng - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (groups[mid].tile_begin <= t) lo = mid; else hi = mid - 1;
  }
  const GemmGroup& G = groups[lo];
  const int64_t local = t - G.tile_begin;
  const int per = G.sym ? G.tiles_per_mat : G.tiles_m * G.tiles_n;
  const int b = static_cast<int>(local / per);
  const int rem = static_cast<int>(local - static_cast<int64_t>(b) * per);
  int mt, nt;
  if (G.sym) {
    const int packed = __ldg(G.tile_list + rem);
    mt = packed >> 16;
    nt = packed & 0xffff;
  } else {
    const int full_panels = G.tiles_n / kPanel;
    const int panel_tiles = G.tiles_m * kPanel;
    const int p = rem / panel_tiles;
    if (p < full_panels) {
      const int within = rem - p * panel_tiles;
      mt = within / kPanel;
      nt = p * kPanel + (within - mt * kPanel);
    } else {
      const int w = G.tiles_n - full_panels * kPanel;
      const int within = rem - full_panels * panel_tiles;
      mt = within / w;
      nt = full_panels * kPanel + (within - mt * w);
    }
  }
  return {lo, b, mt * TILE_M, nt * BN};
}

template <bool FP16>
struct Elem;
template <>
struct Elem<false> {
  using T = __nv_bfloat16;
  __device__ static __forceinline__ float to_f(T v) { return __bfloat162float(v); }
  __device__ static __forceinline__ T from_f(float v) { return __float2bfloat16_rn(v); }
  __device__ static __forceinline__ float bits_to_f(uint16_t v) { return __bfloat162float(__ushort_as_bfloat16(v)); }
};
template <>
struct Elem<true> {
  using T = __half;
  __device__ static __forceinline__ float to_f(T v) { return __half2float(v); }
  __device__ static __forceinline__ T from_f(float v) { return __float2half_rn(v); }
  __device__ static __forceinline__ float bits_to_f(uint16_t v) { return __half2float(__ushort_as_half(v)); }
};

// A bounded wait expired: the other roles of the CTA give up at their next wait, and the
// status word records where (kernel, role, barrier) unless an earlier expiry is there.
template <int STAGES>
__device__ __forceinline__ void signal_timeout(Ctrl<STAGES>* ctrl, int* status, int kernel, int role,
                                               int site) {
  ctrl->abort = 1;
  record_timeout(status, kernel, role, site);
}

// Epilogue of one accumulator: this warp's 32 rows (rows rb .. rb+31 of the matrix,
// TMEM lanes 32*quarter ..), the tile's n_len columns from column n0.
// Two values rounded to the storage format and packed into one 32-bit word (the first
// in the low half), with one conversion instruction.
template <bool FP16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi);
template <>
__device__ __forceinline__ uint32_t pack2<true>(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <>
__device__ __forceinline__ uint32_t pack2<false>(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// 16-bit element j of a packed row (element 2i in the low half of word i).
__device__ __forceinline__ uint16_t half_of(const uint32_t (&h)[16], int j) {
  return static_cast<uint16_t>((j & 1) ? (h[j >> 1] >> 16) : (h[j >> 1] & 0xffffu));
}

// Factor of a product that reads the chain's stored input X = s U, kept as U 2^k: the
// matrix's s 2^-k (squared for X X^T) multiplies alpha and beta; 1 for every other product
// (times 1 leaves every value as it is).
__device__ __forceinline__ float input_factor(const GemmGroup& G, int b) {
  if (G.in_pow == 0) return 1.f;
  const float x = G.in_scale[b];
  return G.in_pow == 2 ? x * x : x;
}

// v = alpha acc (+ beta aux) (+ diag on the diagonal) for one 32-column chunk of this
// lane's row.
template <bool FP16, bool HAS_AUX>
__device__ __forceinline__ void chunk_values(const uint32_t (&r)[32], const typename Elem<FP16>::T* aux_row,
                                             bool row_ok, int col0, bool full, int n_len, int d, float alpha,
                                             float beta, float diag, float (&v)[32]) {
  using E = Elem<FP16>;
  using T = typename E::T;
  if (alpha == 1.0f) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = alpha * __uint_as_float(r[j]);
  }
  if (HAS_AUX && row_ok) {  // rows past M have no aux row
    if (full) {
      const uint4* src = reinterpret_cast<const uint4*>(aux_row + col0);
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        uint4 pk = __ldg(src + w);
        const T* e = reinterpret_cast<const T*>(&pk);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[w * 8 + j] += beta * E::to_f(e[j]);
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (col0 + j < n_len) v[j] += beta * E::to_f(aux_row[col0 + j]);
      }
    }
  }
  if (diag != 0.0f) {
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (d == j) v[j] += diag;
    }
  }
}

// Bounds tests of the checked build (bounds_ok; compiled out otherwise).  box_in: a TMA
// box whose first element (x innermost, y, batch b) lies inside an x_ext x y_ext matrix of
// a group of `count`, x on a 16-byte boundary.  A is M x K (x = k, y = row), K-major B is
// N x K (x = k, y = column of the product), MN-major B is K x N (x = column, y = k), the
// output M x N (x = column, y = row).  elem_in: a run of w elements from (row, col) of an
// M x N matrix; a run read or written as 16-byte vectors (vec) must also start on a
// 16-byte boundary (`at` is its first element's index in its buffer).
__device__ __forceinline__ bool box_in(int x, int x_ext, int y, int y_ext, int b, int count) {
  return x >= 0 && x < x_ext && (x & 7) == 0 && y >= 0 && y < y_ext && b >= 0 && b < count;
}

__device__ __forceinline__ bool elem_in(int row, int col, int w, int M, int N, int b, int count, int64_t at,
                                        bool vec) {
  return row >= 0 && row < M && col >= 0 && col + w <= N && b >= 0 && b < count && (!vec || (at & 7) == 0);
}

// Where the epilogue records a failed bounds test: the status word and the kernel.
struct Chk {
  int* status;
  int kernel;
};

// Epilogue of a stored product whose rows are not a whole number of 16-byte units (the
// TMA store path needs that): out = alpha acc + beta aux + diag I, rounded once and stored
// by each lane for its row.  A symmetric output stores its upper triangle directly and
// mirrors the strict upper triangle: the warp's 32 x 32 block is transposed through
// shared memory (32 rows of 17 words) as packed 16-bit pairs.
template <bool FP16, bool HAS_AUX>
__device__ __forceinline__ void epilogue_rows_direct(const GemmGroup& G, int b, int rb, int n0, int n_len,
                                                     uint32_t t_row, uint32_t* xw, int lane, float alpha,
                                                     float beta, float diag, bool mirror, Chk chk) {
  using E = Elem<FP16>;
  using T = typename E::T;
  const int row = rb + lane;
  const bool row_ok = row < G.M;
  const int nchunks = (n_len + 31) >> 5;
  T* out_row = reinterpret_cast<T*>(G.out) + static_cast<int64_t>(b) * G.out_bstride +
               static_cast<int64_t>(row) * G.ld_out + n0;
  const T* aux_row = nullptr;
  if (HAS_AUX) {
    aux_row = reinterpret_cast<const T*>(G.aux) + static_cast<int64_t>(b) * G.aux_bstride +
              static_cast<int64_t>(row) * G.ld_aux + n0;
  }
  const int first_col = G.sym ? row : 0;  // a symmetric output stores columns >= row
  for (int c = 0; c < nchunks; ++c) {
    uint32_t r[32];
    __syncwarp();  // tcgen05.ld is warp-aligned: all 32 lanes arrive together
    ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(c * 32), r);
    ptx::tmem_ld_wait();
    const int col0 = c * 32;
    const int gc0 = n0 + col0;
    const bool full = col0 + 32 <= n_len;
    uint32_t h[16];
    {
      float v[32];
      // the aux row's elements of this chunk: 32 as four 16-byte vectors, or the ones in range
      const bool aux_ok =
          !HAS_AUX || !row_ok ||
          bounds_ok(elem_in(row, gc0, full ? 32 : min(32, n_len - col0), G.M, G.N, b, G.count,
                            static_cast<int64_t>(b) * G.aux_bstride + static_cast<int64_t>(row) * G.ld_aux + gc0, full),
                    chk.status, chk.kernel, NSM_ROLE_EPILOGUE, NSM_SITE_AUX);
      chunk_values<FP16, HAS_AUX>(r, aux_row, row_ok && aux_ok, col0, full, n_len, row - gc0, alpha, beta, diag, v);
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] = pack2<FP16>(v[2 * i], v[2 * i + 1]);
    }
    if (row_ok) {
      uint16_t* o16 = reinterpret_cast<uint16_t*>(out_row + col0);
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (col0 + j < n_len && gc0 + j >= first_col &&
            bounds_ok(elem_in(row, gc0 + j, 1, G.M, G.N, b, G.count, 0, false), chk.status, chk.kernel, NSM_ROLE_EPILOGUE,
                      NSM_SITE_OUT)) {
          o16[j] = half_of(h, j);
        }
      }
    }
    if (G.sym && mirror && gc0 + 31 > rb) {
      // lanes whose row is out of range hold values that the row mask below never stores
#pragma unroll
      for (int i = 0; i < 16; ++i) xw[lane * 17 + i] = h[i];
      __syncwarp();
      // lane l gathers column gc0 + l: rows 2i and 2i + 1 from two words, its half of each
      const int wc = lane >> 1;
      const uint32_t sel = (lane & 1) ? 0x7632u : 0x5410u;
      uint32_t m[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) m[i] = __byte_perm(xw[(2 * i) * 17 + wc], xw[(2 * i + 1) * 17 + wc], sel);
      const int mr = gc0 + lane;
      if (mr < G.N && col0 + lane < n_len) {
        uint16_t* m16 = reinterpret_cast<uint16_t*>(reinterpret_cast<T*>(G.out) +
                                                    static_cast<int64_t>(b) * G.out_bstride +
                                                    static_cast<int64_t>(mr) * G.ld_out + rb);
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (rb + j < G.M && mr > rb + j &&
              bounds_ok(elem_in(mr, rb + j, 1, G.M, G.N, b, G.count, 0, false), chk.status, chk.kernel, NSM_ROLE_EPILOGUE,
                        NSM_SITE_OUT)) {
            m16[j] = half_of(m, j);
          }
        }
      }
      __syncwarp();
    }
  }
}

// Byte offset of 16-bit element (row, col) of a 32 x 32 block staged for a TMA store
// with 64-byte swizzle: 64-byte rows, the 16-byte unit index XOR (row / 2) mod 4.
__device__ __forceinline__ uint32_t sw64(int row, int col) {
  return static_cast<uint32_t>(row * 64 + ((((col >> 3) ^ (row >> 1)) & 3) << 4) + (col & 7) * 2);
}

// Epilogue of a stored product: out = alpha acc + beta aux + diag I, rounded once.  The
// warp stages each 32 x 32 block of its rows in shared memory and one lane stores it
// with a TMA store (full lines into L2, instead of 16-byte pieces of 32 rows per store
// instruction).  A symmetric output stores the blocks on and above the diagonal: an
// upper block is also staged transposed and stored at the mirrored position, and the
// diagonal block is completed from its own upper triangle before its store.  Every
// element is written once.  Two slots of 4 KB (block + transposed block) alternate;
// `nst` counts the warp's store groups.
template <bool FP16, bool HAS_AUX>
__device__ __forceinline__ void epilogue_rows(const GemmGroup& G, int b, int rb, int n0, int n_len,
                                              uint32_t t_row, uint32_t stage, uint32_t& nst, int lane,
                                              float alpha, float beta, float diag, bool mirror, Chk chk) {
  using E = Elem<FP16>;
  using T = typename E::T;
  if (rb >= G.M) return;  // the warp's rows are past the matrix
  const int row = rb + lane;
  const bool row_ok = row < G.M;
  const int nchunks = (n_len + 31) >> 5;
  // aux block of a chunk, read coalesced: lane l holds 16-byte unit (l & 3) of row
  // rb + 8w + (l >> 2) for w < 4, one chunk ahead of its use
  const T* aux_blk = nullptr;
  uint4 ax_next[4];
  auto aux_load = [&](int c, uint4 (&ax)[4]) {
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int r = rb + 8 * w + (lane >> 2);
      const int col = 32 * c + 8 * (lane & 3);
      const bool in = r < G.M && col < n_len &&
                      bounds_ok(elem_in(r, n0 + col, 8, G.M, G.N, b, G.count,
                                        static_cast<int64_t>(b) * G.aux_bstride + static_cast<int64_t>(r) * G.ld_aux +
                                            n0 + col,
                                        true),
                                chk.status, chk.kernel, NSM_ROLE_EPILOGUE, NSM_SITE_AUX);
      ax[w] = in ? __ldg(reinterpret_cast<const uint4*>(aux_blk + static_cast<int64_t>(8 * w + (lane >> 2)) * G.ld_aux + col))
                 : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  if (HAS_AUX) {
    aux_blk = reinterpret_cast<const T*>(G.aux) + static_cast<int64_t>(b) * G.aux_bstride +
              static_cast<int64_t>(rb) * G.ld_aux + n0;
    int c = 0;
    while (c < nchunks && G.sym && n0 + 32 * c < rb) ++c;
    if (c < nchunks) aux_load(c, ax_next);
  }
  for (int c = 0; c < nchunks; ++c) {
    const int col0 = c * 32;
    const int gc0 = n0 + col0;  // first column of this block in the matrix
    if (G.sym && gc0 < rb) continue;  // below the diagonal: written as the mirror of its upper block
    const bool diag_blk = G.sym && gc0 == rb;
    const bool upper_blk = G.sym && mirror && gc0 > rb;  // stored again at its mirror image
    const uint32_t slot = stage + (nst & 1u) * 4096u;
    if (nst >= 2 && lane == 0) ptx::bulk_wait_group_read<1>();  // the store two blocks back has read it
    __syncwarp();
    uint4 ax_row[4];  // this lane's aux row of the block
    if (HAS_AUX) {
      uint4 ax[4];
#pragma unroll
      for (int w = 0; w < 4; ++w) ax[w] = ax_next[w];
      if (c + 1 < nchunks) aux_load(c + 1, ax_next);
      // through the slot's first half: row r, unit u at sw64(r, 8u)
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int r = 8 * w + (lane >> 2), u = lane & 3;
        ptx::st_shared_v4(slot + sw64(r, 8 * u), ax[w].x, ax[w].y, ax[w].z, ax[w].w);
      }
      __syncwarp();
#pragma unroll
      for (int u = 0; u < 4; ++u) ax_row[u] = ptx::ld_shared_v4(slot + sw64(lane, 8 * u));
      __syncwarp();  // the slot is rewritten with the output below
    }
    uint32_t r[32];
    __syncwarp();  // tcgen05.ld is warp-aligned: all 32 lanes arrive together
    ptx::tmem_ld_32x32b_x32(t_row + static_cast<uint32_t>(col0), r);
    ptx::tmem_ld_wait();
    uint32_t h[16];
    {
      float v[32];
      if (alpha == 1.0f) {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = alpha * __uint_as_float(r[j]);
      }
      if (HAS_AUX) {
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const T* e = reinterpret_cast<const T*>(&ax_row[u]);
#pragma unroll
          for (int j = 0; j < 8; ++j) v[u * 8 + j] += beta * E::to_f(e[j]);
        }
      }
      if (diag != 0.0f) {
        const int d = row - gc0;
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (d == j) v[j] += diag;
        }
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] = pack2<FP16>(v[2 * i], v[2 * i + 1]);
    }
    (void)row_ok;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ptx::st_shared_v4(slot + static_cast<uint32_t>(lane * 64 + (((u ^ (lane >> 1)) & 3) << 4)), h[4 * u],
                        h[4 * u + 1], h[4 * u + 2], h[4 * u + 3]);
    }
    if (diag_blk) {
      // strictly lower elements (j, lane), j > lane, are this lane's (lane, j)
      __syncwarp();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (j > lane) ptx::st_shared_u16(slot + sw64(j, lane), half_of(h, j));
      }
    } else if (upper_blk) {
      // transposed block: its row j is column j of this block
#pragma unroll
      for (int j = 0; j < 32; ++j) ptx::st_shared_u16(slot + 2048u + sw64(j, lane), half_of(h, j));
    }
    ptx::fence_proxy_async_smem();  // the TMA engine reads the staged blocks next
    __syncwarp();
    if (lane == 0) {
      if (bounds_ok(box_in(gc0, G.N, rb, G.M, b, G.count), chk.status, chk.kernel, NSM_ROLE_EPILOGUE, NSM_SITE_OUT)) {
        ptx::tma_store_3d(G.map_out, slot, gc0, rb, b);
      }
      if (upper_blk &&
          bounds_ok(box_in(rb, G.N, gc0, G.M, b, G.count), chk.status, chk.kernel, NSM_ROLE_EPILOGUE, NSM_SITE_OUT)) {
        ptx::tma_store_3d(G.map_out, slot + 2048u, rb, gc0, b);
      }
      ptx::bulk_commit_group();
    }
    ++nst;
  }
}

// ===================================================================== 1-CTA kernel

template <bool B_MN, bool FP16, bool HAS_AUX>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    k_ns_gemm(const GemmGroup* __restrict__ groups, int ng, int64_t total_tiles, float alpha,
              float beta, float diag, int* status) {
  constexpr int STAGES = S1_STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* epi_base = smem + size_t(STAGES) * S1_STAGE_BYTES;
  const uint32_t epi_stage = ptx::smem_u32(epi_base);
  auto* ctrl = reinterpret_cast<Ctrl<STAGES>*>(smem + size_t(STAGES) * S1_STAGE_BYTES + EPI_STAGE_BYTES);
  const uint32_t ring = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  auto bar = [&](uint64_t* b) { return ptx::smem_u32(b); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar(&ctrl->full[s]), 1);
      ptx::mbar_init(bar(&ctrl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(bar(&ctrl->acc_full[a]), 1);
      ptx::mbar_init(bar(&ctrl->acc_empty[a]), EPI_WARPS);
    }
    ptx::mbar_init(bar(&ctrl->drain), 1);
    ctrl->abort = 0;
    ctrl->never = 0;
    ptx::fence_mbarrier_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(&ctrl->tmem_base), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // barriers and TMEM are set up; the operands come from the previous kernel of the stream
  grid_dependency_sync();
  release_dependents();
  const uint32_t tmem_base = ctrl->tmem_base;
  volatile int* abort_flag = &ctrl->abort;
  volatile int* never_flag = &ctrl->never;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int fill_parity[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) fill_parity[s] = -1;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const TileCoord tc = decode_tile<128>(groups, ng, t);
        const GemmGroup& G = groups[tc.g];
        const int kblocks = (G.K + BK - 1) / BK;
        const int n_len = min(BN, G.N - tc.n0);
        const int nb = (n_len + 63) >> 6;
        // A: one box of a_box >= 128 rows, or 64-row boxes for the rows in range; B likewise
        // (MN-major B: 64-column boxes of 64 K rows)
        const int a_loads = G.a_box >= 128 ? 1 : ((G.M - tc.m0 > 64) ? 2 : 1);
        const int a_rows = G.a_box >= 128 ? G.a_box : 64;
        const int b_loads = (!B_MN && G.b_box >= 256) ? 1 : nb;
        const int b_rows = (!B_MN && G.b_box >= 256) ? G.b_box : 64;
        const uint32_t bytes = static_cast<uint32_t>((a_loads * a_rows + b_loads * b_rows) * 128);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait_bounded(bar(&ctrl->empty[stage]), phase ^ 1u, abort_flag,
                                      WAIT_LIMIT_NS)) {
            signal_timeout(ctrl, status, NSM_KERNEL_GEMM, NSM_ROLE_PRODUCER, NSM_SITE_STAGE_EMPTY);
            ok = false;
            break;
          }
          const uint32_t fb = bar(&ctrl->full[stage]);
          ptx::mbar_arrive_expect_tx(fb, bytes);
          const uint32_t a_dst = ring + stage * S1_STAGE_BYTES;
          const uint32_t b_dst = a_dst + S1_A_BYTES;
          const int k0 = kb * BK;
          constexpr int K1 = NSM_KERNEL_GEMM, RP = NSM_ROLE_PRODUCER;
          for (int q = 0; q < a_loads; ++q) {
            if (bounds_ok(box_in(k0, G.K, tc.m0 + 64 * q, G.M, tc.b, G.count), status, K1, RP, NSM_SITE_TMA_A)) {
              ptx::tma_load_3d(a_dst + q * BOX_BYTES, G.map_a, fb, k0, tc.m0 + 64 * q, tc.b);
            }
          }
          for (int q = 0; q < b_loads; ++q) {
            if (B_MN) {
              if (bounds_ok(box_in(tc.n0 + 64 * q, G.N, k0, G.K, tc.b, G.count), status, K1, RP, NSM_SITE_TMA_B)) {
                ptx::tma_load_3d(b_dst + q * BOX_BYTES, G.map_b, fb, tc.n0 + 64 * q, k0, tc.b);
              }
            } else {
              if (bounds_ok(box_in(k0, G.K, tc.n0 + 64 * q, G.N, tc.b, G.count), status, K1, RP, NSM_SITE_TMA_B)) {
                ptx::tma_load_3d(b_dst + q * BOX_BYTES, G.map_b, fb, k0, tc.n0 + 64 * q, tc.b);
              }
            }
          }
          fill_parity[stage] = static_cast<int>(phase);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let every copy already issued land before the block can exit.
        for (int s = 0; s < STAGES; ++s) {
          if (fill_parity[s] >= 0) {
            ptx::mbar_wait_bounded(bar(&ctrl->full[s]), static_cast<uint32_t>(fill_parity[s]),
                                   never_flag, WAIT_LIMIT_NS);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      for (int64_t t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++local) {
        const TileCoord tc = decode_tile<128>(groups, ng, t);
        const GemmGroup& G = groups[tc.g];
        const int kblocks = (G.K + BK - 1) / BK;
        const int n_len = min(BN, G.N - tc.n0);
        const int nb = (n_len + 63) >> 6;
        const int acc = local & 1;
        const uint32_t acc_phase = static_cast<uint32_t>((local >> 1) & 1);
        if (!ptx::mbar_wait_bounded(bar(&ctrl->acc_empty[acc]), acc_phase ^ 1u, abort_flag,
                                    WAIT_LIMIT_NS)) {
          signal_timeout(ctrl, status, NSM_KERNEL_GEMM, NSM_ROLE_MMA, NSM_SITE_ACC_EMPTY);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        const uint32_t idesc = ptx::idesc_f16(128, nb * 64, !FP16, B_MN);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait_bounded(bar(&ctrl->full[stage]), phase, abort_flag,
                                      WAIT_LIMIT_NS)) {
            signal_timeout(ctrl, status, NSM_KERNEL_GEMM, NSM_ROLE_MMA, NSM_SITE_STAGE_FULL);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ring + stage * S1_STAGE_BYTES;
          const uint32_t b_addr = a_addr + S1_A_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t a_desc = ptx::smem_desc_sw128(a_addr + kk * 32, 16, 1024);
            const uint64_t b_desc = B_MN ? ptx::smem_desc_sw128(b_addr + kk * 2048, BOX_BYTES, 1024)
                                         : ptx::smem_desc_sw128(b_addr + kk * 32, 16, 1024);
            ptx::mma_f16(d_tmem, a_desc, b_desc, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(bar(&ctrl->empty[stage]));
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit(bar(&ctrl->acc_full[acc]));
      }
      // No MMA may still write TMEM when the block frees it.
      ptx::mma_commit(bar(&ctrl->drain));
      if (!ptx::mbar_wait_bounded(bar(&ctrl->drain), 0u, never_flag, WAIT_LIMIT_NS)) {
        signal_timeout(ctrl, status, NSM_KERNEL_GEMM, NSM_ROLE_TEARDOWN, NSM_SITE_DRAIN);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;  // TMEM lanes this warp may access: 32*quarter + [0, 32)
    const uint32_t stage = epi_stage + static_cast<uint32_t>(warp - 2) * 8192u;  // 1024-byte aligned
    uint32_t* stage_words = reinterpret_cast<uint32_t*>(epi_base + (warp - 2) * 8192);
    uint32_t nst = 0;
    int local = 0;
    for (int64_t t = blockIdx.x; t < total_tiles; t += gridDim.x, ++local) {
      const TileCoord tc = decode_tile<128>(groups, ng, t);
      const GemmGroup& G = groups[tc.g];
      const int acc = local & 1;
      const uint32_t acc_phase = static_cast<uint32_t>((local >> 1) & 1);
      bool ok = true;
      if (lane == 0) {
        ok = ptx::mbar_wait_bounded(bar(&ctrl->acc_full[acc]), acc_phase, abort_flag,
                                    WAIT_LIMIT_NS);
        if (!ok) signal_timeout(ctrl, status, NSM_KERNEL_GEMM, NSM_ROLE_EPILOGUE, NSM_SITE_ACC_FULL);
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      const float f = input_factor(G, tc.b);
      if (G.map_out) {
        epilogue_rows<FP16, HAS_AUX>(G, tc.b, tc.m0 + quarter * 32, tc.n0, min(BN, G.N - tc.n0),
                                     t_row, stage, nst, lane, alpha * f, beta * f, diag, true,
                                     Chk{status, NSM_KERNEL_GEMM});
      } else {
        epilogue_rows_direct<FP16, HAS_AUX>(G, tc.b, tc.m0 + quarter * 32, tc.n0, min(BN, G.N - tc.n0),
                                            t_row, stage_words, lane, alpha * f, beta * f, diag, true,
                                            Chk{status, NSM_KERNEL_GEMM});
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(&ctrl->acc_empty[acc]));
    }
    // staged blocks must be read out by the TMA engine before the block exits
    if (lane == 0) ptx::bulk_wait_group<0>();
    __syncwarp();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

// ===================================================================== pair kernel
//
// A cluster of two CTAs (ranks 0 and 1, the leader is rank 0) owns one 256 x 256 output
// tile at a time.  Rank r stages rows [m0 + 128r, +128) of A and rows (K-major B) or
// columns (MN-major B) [n0 + 128r, +128) of B; its TMA loads count on the leader's full
// barrier.  The leader issues tcgen05.mma.cta_group::2 (M = 256, N = 256) and commits to
// both CTAs' empty / accumulator barriers with a multicast.  Each CTA's TMEM receives its
// own 128 rows of D; the epilogue warps of both CTAs arrive on the leader's
// accumulator-empty barrier.  Every wait is bounded; every path reaches the closing
// cluster barrier.

__device__ __forceinline__ int boxes_in(int start, int limit) {
  // 64-wide boxes of the 128-wide half starting at `start` that hold any in-range index
  const int left = limit - start;
  return left <= 0 ? 0 : (left > 64 ? 2 : 1);
}

template <bool B_MN, bool FP16, bool HAS_AUX, bool NARROW>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    k_ns_gemm_pair(const GemmGroup* __restrict__ groups, int ng, int64_t total_tiles, float alpha,
                   float beta, float diag, int* status) {
  constexpr int STAGES = S2_STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* epi_base = smem + size_t(STAGES) * S2_STAGE_BYTES;
  const uint32_t epi_stage = ptx::smem_u32(epi_base);
  auto* ctrl = reinterpret_cast<Ctrl<STAGES>*>(smem + size_t(STAGES) * S2_STAGE_BYTES + EPI_STAGE_BYTES);
  const uint32_t ring = ptx::smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int64_t pair = blockIdx.x >> 1;
  const int64_t npairs = gridDim.x >> 1;

  auto bar = [&](uint64_t* b) { return ptx::smem_u32(b); };

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(bar(&ctrl->full[s]), 1);
      ptx::mbar_init(bar(&ctrl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(bar(&ctrl->acc_full[a]), 1);
      ptx::mbar_init(bar(&ctrl->acc_empty[a]), 2 * EPI_WARPS);
    }
    ptx::mbar_init(bar(&ctrl->drain), 1);
    ctrl->abort = 0;
    ctrl->never = 0;
    ptx::fence_mbarrier_init();
  }
  // both CTAs' barriers must exist before either CTA signals the other's
  ptx::cluster_sync();
  if (warp == 0) {
    ptx::tmem_alloc_pair(ptx::smem_u32(&ctrl->tmem_base), TMEM_COLS);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // barriers and TMEM are set up; the operands come from the previous kernel of the stream
  grid_dependency_sync();
  release_dependents();
  const uint32_t tmem_base = ctrl->tmem_base;
  volatile int* abort_flag = &ctrl->abort;
  volatile int* never_flag = &ctrl->never;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int fill_parity[STAGES];
#pragma unroll
      for (int s = 0; s < STAGES; ++s) fill_parity[s] = -1;
      bool ok = true;
      for (int64_t t = pair; t < total_tiles && ok; t += npairs) {
        const TileCoord tc = decode_tile<256>(groups, ng, t);
        const GemmGroup& G = groups[tc.g];
        const int kblocks = (G.K + BK2 - 1) / BK2;
        // boxes each CTA loads; the leader expects both CTAs' bytes
        const int a0 = boxes_in(tc.m0, G.M), a1 = boxes_in(tc.m0 + 128, G.M);
        // A tile with at most 128 columns in range runs N = 128 MMAs: each CTA then stages
        // 64 columns of B (rank r: [n0 + 64r, +64)), one 64-wide box, instead of 128.  Only
        // the instance for launches that have such tiles (NARROW) tests for them.
        const bool narrow = NARROW && G.N - tc.n0 <= 128;
        const int b0 = narrow ? 1 : boxes_in(tc.n0, G.N);
        const int b1 = narrow ? (tc.n0 + 64 < G.N ? 1 : 0) : boxes_in(tc.n0 + 128, G.N);
        // Per 64-wide K box, a K-major half with any row in range loads one box of 128 rows
        // (a_box / b_box >= 128) or one 64-row box per 64 rows in range.  An MN-major B half
        // loads one box per 64 columns in range, each holding the stage's K rows (b_box =
        // 128 K rows, or 64 with one box per K box).
        auto loads = [](int units, int box) { return box >= 128 ? (units ? 1 : 0) : units; };
        auto rows = [](int box) { return box >= 128 ? box : 64; };
        const int my_a = loads(rank ? a1 : a0, G.a_box);
        const int my_b = (B_MN || narrow) ? (rank ? b1 : b0) : loads(rank ? b1 : b0, G.b_box);
        const uint32_t a_bytes_k = static_cast<uint32_t>((loads(a0, G.a_box) + loads(a1, G.a_box)) * rows(G.a_box) * 128);
        const uint32_t b_bytes_k = static_cast<uint32_t>(
            (B_MN || narrow) ? (b0 + b1) * 64 * 128 : (loads(b0, G.b_box) + loads(b1, G.b_box)) * rows(G.b_box) * 128);
        const int row0 = tc.m0 + 128 * static_cast<int>(rank);
        const int col0 = tc.n0 + (narrow ? 64 : 128) * static_cast<int>(rank);
        const CUtensorMap* map_b = narrow ? G.map_b_narrow : G.map_b;
        // Operands stored as upper 256 x 256 tiles: a K block before the operand's own tile
        // (mt for A, nt for B) lies below the diagonal, and is loaded from its mirror image
        // as an MN-major operand: one 64-column box of 128 K rows per 64 rows (A) or
        // columns (B) in range, through the same maps (boxes of 64 x 128).
        const int mt = tc.m0 >> 8, nt = tc.n0 >> 8;
        const bool lean_a = (G.lean & kLeanA) != 0;
        const bool lean_b = !B_MN && (G.lean & kLeanB) != 0;
        const int my_at = rank ? a1 : a0;
        const int my_bt = rank ? b1 : b0;
        const uint32_t a_bytes_t = static_cast<uint32_t>((a0 + a1) * 2 * BOX_BYTES);
        const uint32_t b_bytes_t = static_cast<uint32_t>((b0 + b1) * 2 * BOX_BYTES);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait_bounded(bar(&ctrl->empty[stage]), phase ^ 1u, abort_flag,
                                      WAIT_LIMIT_NS)) {
            signal_timeout(ctrl, status, NSM_KERNEL_GEMM_PAIR, NSM_ROLE_PRODUCER, NSM_SITE_STAGE_EMPTY);
            ok = false;
            break;
          }
          const uint32_t fb_local = bar(&ctrl->full[stage]);
          const uint32_t fb_leader = ptx::mapa_shared(fb_local, 0);
          const int k0 = kb * BK2;
          const int nk = (G.K - k0 > 64) ? 2 : 1;  // 64-wide K boxes holding any K in range
          // MN-major B boxes with 128 K rows load both K boxes at once
          const int b_k_loads = (B_MN && G.b_box >= 128) ? 1 : nk;
          const bool at = lean_a && (kb >> 1) < mt;  // this stage's 256-wide K tile is kb / 2
          const bool bt = lean_b && (kb >> 1) < nt;
          const uint32_t bytes = (at ? a_bytes_t : a_bytes_k * nk) +
                                 (B_MN ? (G.b_box >= 128 ? 2 * b_bytes_k : b_bytes_k * nk)
                                       : (bt ? b_bytes_t : b_bytes_k * nk));
          if (rank == 0) ptx::mbar_arrive_expect_tx(fb_local, bytes);
          // stage layout: A [K box][128 rows]; K-major B [K box][128 rows];
          // MN-major A or B [64-column block][128 K rows]
          const uint32_t a_dst = ring + stage * S2_STAGE_BYTES;
          const uint32_t b_dst = a_dst + S2_A_BYTES;
          constexpr int K2 = NSM_KERNEL_GEMM_PAIR, RP = NSM_ROLE_PRODUCER;
          if (at) {
            for (int q = 0; q < my_at; ++q) {
              if (bounds_ok(box_in(row0 + 64 * q, G.M, k0, G.K, tc.b, G.count), status, K2, RP, NSM_SITE_TMA_A)) {
                ptx::tma_load_3d_pair(a_dst + q * 2 * BOX_BYTES, G.map_a, fb_leader, row0 + 64 * q, k0, tc.b);
              }
            }
          } else {
            for (int kq = 0; kq < nk; ++kq) {
              for (int q = 0; q < my_a; ++q) {
                if (bounds_ok(box_in(k0 + 64 * kq, G.K, row0 + 64 * q, G.M, tc.b, G.count), status, K2, RP,
                              NSM_SITE_TMA_A)) {
                  ptx::tma_load_3d_pair(a_dst + kq * 2 * BOX_BYTES + q * BOX_BYTES, G.map_a, fb_leader,
                                        k0 + 64 * kq, row0 + 64 * q, tc.b);
                }
              }
            }
          }
          if (!B_MN && bt) {
            for (int q = 0; q < my_bt; ++q) {
              if (bounds_ok(box_in(col0 + 64 * q, G.N, k0, G.K, tc.b, G.count), status, K2, RP, NSM_SITE_TMA_B)) {
                ptx::tma_load_3d_pair(b_dst + q * 2 * BOX_BYTES, G.map_b, fb_leader, col0 + 64 * q, k0, tc.b);
              }
            }
          } else if (!B_MN) {
            for (int kq = 0; kq < nk; ++kq) {
              for (int q = 0; q < my_b; ++q) {
                if (bounds_ok(box_in(k0 + 64 * kq, G.K, col0 + 64 * q, G.N, tc.b, G.count), status, K2, RP,
                              NSM_SITE_TMA_B)) {
                  ptx::tma_load_3d_pair(b_dst + kq * 2 * BOX_BYTES + q * BOX_BYTES, map_b, fb_leader,
                                        k0 + 64 * kq, col0 + 64 * q, tc.b);
                }
              }
            }
          }
          if (B_MN) {
            for (int kq = 0; kq < b_k_loads; ++kq) {
              for (int q = 0; q < my_b; ++q) {
                if (bounds_ok(box_in(col0 + 64 * q, G.N, k0 + 64 * kq, G.K, tc.b, G.count), status, K2, RP,
                              NSM_SITE_TMA_B)) {
                  ptx::tma_load_3d_pair(b_dst + q * 2 * BOX_BYTES + kq * BOX_BYTES, map_b, fb_leader,
                                        col0 + 64 * q, k0 + 64 * kq, tc.b);
                }
              }
            }
          }
          fill_parity[stage] = static_cast<int>(phase);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        if (rank == 0) {
          // the leader's full barriers count both CTAs' copies: wait for those in flight
          for (int s = 0; s < STAGES; ++s) {
            if (fill_parity[s] >= 0) {
              ptx::mbar_wait_bounded(bar(&ctrl->full[s]), static_cast<uint32_t>(fill_parity[s]),
                                     never_flag, WAIT_LIMIT_NS);
            }
          }
        } else {
          // the peer cannot observe the leader's barriers: give its copies time to land
          const uint64_t t0 = ptx::globaltimer_ns();
          while (ptx::globaltimer_ns() - t0 < 1000000ull) {
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (leader)
    if (lane == 0 && rank == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int local = 0;
      bool ok = true;
      const uint32_t idesc_wide = ptx::idesc_f16(256, 256, !FP16, B_MN);
      const uint32_t idesc_narrow = ptx::idesc_f16(256, 128, !FP16, B_MN);
      for (int64_t t = pair; t < total_tiles && ok; t += npairs, ++local) {
        const TileCoord tc = decode_tile<256>(groups, ng, t);
        const GemmGroup& G = groups[tc.g];
        const int kblocks = (G.K + BK2 - 1) / BK2;
        // at most 128 columns in range: N = 128, each CTA's B holds 64 of them
        const uint32_t idesc = (NARROW && G.N - tc.n0 <= 128) ? idesc_narrow : idesc_wide;
        // K blocks below the diagonal of an operand stored as upper tiles arrive MN-major
        const int mt = tc.m0 >> 8, nt = tc.n0 >> 8;
        const bool lean_a = (G.lean & kLeanA) != 0;
        const bool lean_b = !B_MN && (G.lean & kLeanB) != 0;
        const int acc = local & 1;
        const uint32_t acc_phase = static_cast<uint32_t>((local >> 1) & 1);
        if (!ptx::mbar_wait_bounded(bar(&ctrl->acc_empty[acc]), acc_phase ^ 1u, abort_flag,
                                    WAIT_LIMIT_NS)) {
          signal_timeout(ctrl, status, NSM_KERNEL_GEMM_PAIR, NSM_ROLE_MMA, NSM_SITE_ACC_EMPTY);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < kblocks; ++kb) {
          if (!ptx::mbar_wait_bounded(bar(&ctrl->full[stage]), phase, abort_flag,
                                      WAIT_LIMIT_NS)) {
            signal_timeout(ctrl, status, NSM_KERNEL_GEMM_PAIR, NSM_ROLE_MMA, NSM_SITE_STAGE_FULL);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a_addr = ring + stage * S2_STAGE_BYTES;
          const uint32_t b_addr = a_addr + S2_A_BYTES;
          // K slices of 16 in range (the last stage may hold fewer than 8)
          const int left = G.K - kb * BK2;
          const int nslices = left >= BK2 ? BK2 / 16 : (left + 15) / 16;
          const bool at = lean_a && (kb >> 1) < mt;
          const bool bt = B_MN || (lean_b && (kb >> 1) < nt);
          const uint32_t id = idesc | (at ? ptx::kIdescAMajorMN : 0u) | (bt ? ptx::kIdescBMajorMN : 0u);
          for (int kk = 0; kk < nslices; ++kk) {
            const uint32_t koff = static_cast<uint32_t>((kk >> 2) * 2 * BOX_BYTES + (kk & 3) * 32);
            // K-major: 64-wide K boxes of 128 rows, a slice 32 bytes into a row; MN-major:
            // 64-wide row (A) or column (B) blocks 16 KB apart, a slice 16 K rows down
            const uint64_t a_desc = at ? ptx::smem_desc_sw128(a_addr + kk * 2048, 2 * BOX_BYTES, 1024)
                                       : ptx::smem_desc_sw128(a_addr + koff, 16, 1024);
            const uint64_t b_desc = bt ? ptx::smem_desc_sw128(b_addr + kk * 2048, 2 * BOX_BYTES, 1024)
                                       : ptx::smem_desc_sw128(b_addr + koff, 16, 1024);
            ptx::mma_f16_pair(d_tmem, a_desc, b_desc, id, (kb | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit_pair(bar(&ctrl->empty[stage]), 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        ptx::mma_commit_pair(bar(&ctrl->acc_full[acc]), 0x3);
      }
      // both CTAs' drain barriers complete once every MMA of the pair has finished
      ptx::mma_commit_pair(bar(&ctrl->drain), 0x3);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (warps 2..5)
    const int quarter = warp & 3;
    const uint32_t stage = epi_stage + static_cast<uint32_t>(warp - 2) * 8192u;  // 1024-byte aligned
    uint32_t* stage_words = reinterpret_cast<uint32_t*>(epi_base + (warp - 2) * 8192);
    uint32_t nst = 0;
    int local = 0;
    for (int64_t t = pair; t < total_tiles; t += npairs, ++local) {
      const TileCoord tc = decode_tile<256>(groups, ng, t);
      const GemmGroup& G = groups[tc.g];
      const int acc = local & 1;
      const uint32_t acc_phase = static_cast<uint32_t>((local >> 1) & 1);
      bool ok = true;
      if (lane == 0) {
        ok = ptx::mbar_wait_bounded(bar(&ctrl->acc_full[acc]), acc_phase, abort_flag,
                                    WAIT_LIMIT_NS);
        if (!ok) signal_timeout(ctrl, status, NSM_KERNEL_GEMM_PAIR, NSM_ROLE_EPILOGUE, NSM_SITE_ACC_FULL);
      }
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      ptx::tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc * BN);
      const int rb = tc.m0 + 128 * static_cast<int>(rank) + quarter * 32;
      // an output stored as upper 256 x 256 tiles mirrors blocks only inside diagonal tiles
      const bool mirror = !(G.lean & kLeanOut) || tc.m0 == tc.n0;
      const float f = input_factor(G, tc.b);
      if (G.map_out) {
        epilogue_rows<FP16, HAS_AUX>(G, tc.b, rb, tc.n0, min(BN, G.N - tc.n0), t_row, stage, nst, lane,
                                     alpha * f, beta * f, diag, mirror, Chk{status, NSM_KERNEL_GEMM_PAIR});
      } else {
        epilogue_rows_direct<FP16, HAS_AUX>(G, tc.b, rb, tc.n0, min(BN, G.N - tc.n0), t_row, stage_words,
                                            lane, alpha * f, beta * f, diag, mirror, Chk{status, NSM_KERNEL_GEMM_PAIR});
      }
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(ptx::mapa_shared(bar(&ctrl->acc_empty[acc]), 0));
    }
    // staged blocks must be read out by the TMA engine before the block exits
    if (lane == 0) ptx::bulk_wait_group<0>();
    __syncwarp();
  }

  // no MMA of the pair may still write this CTA's TMEM when it is freed
  if (threadIdx.x == 0) {
    if (!ptx::mbar_wait_bounded(bar(&ctrl->drain), 0u, never_flag, WAIT_LIMIT_NS)) {
      signal_timeout(ctrl, status, NSM_KERNEL_GEMM_PAIR, NSM_ROLE_TEARDOWN, NSM_SITE_DRAIN);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  // neither CTA leaves while the other may still signal its barriers
  ptx::cluster_sync();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

// ===================================================================== launchers

template <typename K>
cudaError_t set_smem_once(K kernel, size_t bytes, std::atomic<uint64_t>& done) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!bit || !(done.load() & bit)) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
    done.fetch_or(bit);
  }
  return cudaSuccess;
}

template <bool B_MN, bool FP16, bool HAS_AUX, bool NARROW>
cudaError_t launch_pair(const GemmLaunch& l, int num_sms, cudaStream_t stream, int* status) {
  static std::atomic<uint64_t> done{0};
  static std::atomic<int> max_clusters[64];
  cudaError_t e = set_smem_once(k_ns_gemm_pair<B_MN, FP16, HAS_AUX, NARROW>, S2_SMEM, done);
  if (e != cudaSuccess) return e;
  // as many pairs as can be resident at once (a GPC with an odd number of free SMs
  // cannot host a cluster of two)
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int resident = (dev >= 0 && dev < 64) ? max_clusters[dev].load() : 0;
  if (resident <= 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(num_sms & ~1), 1, 1);
    cfg.blockDim = dim3(NUM_THREADS, 1, 1);
    cfg.dynamicSmemBytes = S2_SMEM;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = 2;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&resident, k_ns_gemm_pair<B_MN, FP16, HAS_AUX, NARROW>, &cfg) != cudaSuccess ||
        resident <= 0) {
      cudaGetLastError();
      resident = num_sms / 2;
    }
    if (dev >= 0 && dev < 64) max_clusters[dev].store(resident);
  }
  const int64_t cap = resident < num_sms / 2 ? resident : num_sms / 2;
  const int64_t pairs = l.total_tiles < cap ? l.total_tiles : cap;
  if (pairs <= 0) return cudaSuccess;
  if (const cudaError_t e_launch = launch_ordered(kOverlapGemmLaunch, k_ns_gemm_pair<B_MN, FP16, HAS_AUX, NARROW>,
                                              dim3(static_cast<unsigned>(2 * pairs)), dim3(NUM_THREADS), S2_SMEM,
                                              stream, l.groups, l.num_groups, l.total_tiles, l.alpha, l.beta, l.diag,
                                              status))
    return e_launch;
  return cudaGetLastError();
}

template <bool B_MN, bool FP16, bool HAS_AUX>
cudaError_t launch_typed(const GemmLaunch& l, int num_sms, cudaStream_t stream) {
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  if (l.pair) {
    return l.narrow ? launch_pair<B_MN, FP16, HAS_AUX, true>(l, num_sms, stream, status)
                    : launch_pair<B_MN, FP16, HAS_AUX, false>(l, num_sms, stream, status);
  }
  static std::atomic<uint64_t> done{0};
  cudaError_t e = set_smem_once(k_ns_gemm<B_MN, FP16, HAS_AUX>, S1_SMEM, done);
  if (e != cudaSuccess) return e;
  const int64_t grid = l.total_tiles < num_sms ? l.total_tiles : num_sms;
  if (grid <= 0) return cudaSuccess;
  if (const cudaError_t e_launch = launch_ordered(kOverlapGemmLaunch, k_ns_gemm<B_MN, FP16, HAS_AUX>, dim3(static_cast<unsigned>(grid)),
                                              dim3(NUM_THREADS), S1_SMEM, stream, l.groups, l.num_groups, l.total_tiles,
                                              l.alpha, l.beta, l.diag, status))
    return e_launch;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm(const GemmLaunch& l, int num_sms, cudaStream_t stream) {
  const int key = (l.b_mn_major ? 4 : 0) | (l.fp16 ? 2 : 0) | (l.has_aux ? 1 : 0);
  switch (key) {
    case 0: return launch_typed<false, false, false>(l, num_sms, stream);
    case 1: return launch_typed<false, false, true>(l, num_sms, stream);
    case 2: return launch_typed<false, true, false>(l, num_sms, stream);
    case 3: return launch_typed<false, true, true>(l, num_sms, stream);
    case 4: return launch_typed<true, false, false>(l, num_sms, stream);
    case 5: return launch_typed<true, false, true>(l, num_sms, stream);
    case 6: return launch_typed<true, true, false>(l, num_sms, stream);
    default: return launch_typed<true, true, true>(l, num_sms, stream);
  }
}

}  // namespace nsm
