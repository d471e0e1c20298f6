// The whole Newton-Schulz chain of small matrices (working m <= 128) in one launch.
//
// "DeepSpeed 集成 Muon 优化器实战" §核心算子 gives the iteration; for a matrix whose short side
// is at most 128, every m x m iterate (A and B of the standard form; R, H, Q and T of the
// gram form) fits one 128 x 128 tile of shared memory (32 KB in 16-bit storage).  One CTA
// runs the chain of one matrix at a time (persistently over the launch's matrices):
//
//   * m x m products  S[dst] = alpha S[a] S[b]^T + beta S[aux] + diag I  read both operands
//     from shared memory (8 MMAs of 128 x 128 x 16) and write the rounded result back
//     there from the TMEM accumulator;
//   * passes over X (m x n, n up to the tensor's width) stream 128-column chunks of X
//     (two 64-column panels each) through a 2-slot TMA ring:
//       Gram:  S[dst] = X X^T, each chunk being both operands (K-major);
//       pass:  X' = alpha S[a] X + beta X, the chunk being the MN-major B operand
//              (N = 128).  Each chunk of X' is rounded in the epilogue, written to
//              shared memory and stored with TMA stores; when another Gram follows, the
//              MMA warp also accumulates X' X'^T from that chunk, so the next step needs
//              no extra pass over X.  The final pass stores O the same way; the step's
//              separate apply pass then updates the parameters (the four epilogue warps
//              of a CTA cannot keep enough parameter loads in flight to apply it here:
//              measured, that took 62% of this kernel's time on the Split/MoE head blocks).
//
// Roles: warp 0 issues the TMA loads, warp 1 (one thread) the MMAs, warps 2-5 drain TMEM
// (each thread one row).  Every wait is bounded; the epilogue warps take every decision
// to give up together (a barrier reduction), so no warp is left at a named barrier.
// Every m x m iterate is symmetric (a polynomial in X X^T), which is why S[b]^T serves
// for S[b] and one K-major layout serves every use.  The chain's input is stored as U 2^k;
// the Gram and pass operations that read it take the matrix's s 2^-k into alpha and beta
// (squared for the Gram), so that they compute with X = s U.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>

#include "launch.cuh"
#include "nsm_internal.h"
#include "ptx.cuh"

namespace nsm {
namespace {

constexpr int kThreads = 192;
constexpr int kPanel = 128 * 128;          // 128 rows x 64 16-bit columns, 128-byte swizzle
constexpr int kSquare = 2 * kPanel;        // 128 x 128: two 64-column panels
constexpr int kSquares = 3;
constexpr int kChunk = 128;                // columns of X per pass step: two panels
constexpr int kSlot = 2 * kPanel;          // one chunk in shared memory (the layout of a square)
constexpr int kRing = 2;                   // chunk slots of the TMA ring
constexpr uint32_t kTmemCols = 512;        // [0,128) m x m accumulator; [128,384) two chunk accumulators
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr uint32_t kEpiBar = 1;            // named barrier of the epilogue warps
constexpr uint32_t kEpiThreads = 128;

struct Ctrl {
  uint64_t full[kRing];
  uint64_t empty[kRing];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint64_t xt_full[2];
  uint64_t xt_empty[2];
  uint64_t sq_full;
  uint64_t sq_done;
  uint64_t stores_done;
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
  int never;
};

constexpr size_t kRingOff = size_t(kSquares) * kSquare;
constexpr size_t kXtOff = kRingOff + size_t(kRing) * kSlot;
constexpr size_t kCtrlOff = kXtOff + 2 * size_t(kSlot);
constexpr size_t kSmem = 1024 + kCtrlOff + sizeof(Ctrl);
static_assert(kSmem <= 232448, "shared memory per CTA");

template <bool FP16>
struct Store;
template <>
struct Store<false> {
  using T = __nv_bfloat16;
  __device__ static __forceinline__ float to_f(T v) { return __bfloat162float(v); }
  __device__ static __forceinline__ T from_f(float v) { return __float2bfloat16_rn(v); }
};
template <>
struct Store<true> {
  using T = __half;
  __device__ static __forceinline__ float to_f(T v) { return __half2float(v); }
  __device__ static __forceinline__ T from_f(float v) { return __float2half_rn(v); }
};

// Byte offset of 16-byte unit u (0..7) of row `row` in a 128-byte-swizzled panel.
__device__ __forceinline__ uint32_t sw(int row, int u) {
  return static_cast<uint32_t>(row * 128 + ((u ^ (row & 7)) << 4));
}

// K-major descriptor of K-slice kk (16 columns) of a 128 x 128 shared-memory matrix.
__device__ __forceinline__ uint64_t square_desc(uint32_t base, int kk) {
  return ptx::smem_desc_sw128(base + static_cast<uint32_t>((kk >> 2) * kPanel + (kk & 3) * 32), 16, 1024);
}

struct Roles {
  Ctrl* ctrl;
  uint32_t squares, ring, xt;
  int* status;
  volatile int* abort_flag;
  volatile int* never_flag;

  __device__ uint32_t bar(uint64_t* b) const { return ptx::smem_u32(b); }
  __device__ uint32_t square(int i) const { return squares + static_cast<uint32_t>(i * kSquare); }
  // Bounded wait; on expiry the status word records this role and barrier (unless an
  // earlier expiry is there) and the other roles give up at their next wait.
  __device__ bool wait(uint64_t* b, uint32_t parity, int role, int site) const {
    if (ptx::mbar_wait_bounded(bar(b), parity, abort_flag, kWaitNs)) return true;
    if (!*abort_flag) record_timeout(status, NSM_KERNEL_SMALL, role, site);
    ctrl->abort = 1;
    return false;
  }
  __device__ void give_up() const { ctrl->abort = 1; }
};

struct RingPos {
  int stage = 0;
  uint32_t phase = 0;
  __device__ void advance() {
    if (++stage == kRing) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

// ------------------------------------------------------------------ TMA producer
__device__ bool produce(const Roles& R, const SmallJob* __restrict__ jobs, int njobs,
                        const SmallOp* __restrict__ ops, int nops, int (&fill_parity)[kRing]) {
  RingPos rp;
  uint32_t stores_seen = 0;
  for (int j = blockIdx.x; j < njobs; j += gridDim.x) {
    const SmallJob job = jobs[j];
    const int nck = (job.n + kChunk - 1) / kChunk;
    bool first_pass = true;
    for (int o = 0; o < nops; ++o) {
      const SmallOp op = ops[o];
      if (op.kind == kSmallSquare) continue;
      if (op.kind == kSmallPass) {
        // the source was stored by the previous pass of this matrix: wait until it landed
        if (!first_pass) {
          if (!R.wait(&R.ctrl->stores_done, stores_seen & 1u, NSM_ROLE_PRODUCER, NSM_SITE_STORES_DONE)) return false;
          ++stores_seen;
        }
        first_pass = false;
      }
      const CUtensorMap* map = job.map_x[op.src_x];
      for (int c = 0; c < nck; ++c) {
        if (!R.wait(&R.ctrl->empty[rp.stage], rp.phase ^ 1u, NSM_ROLE_PRODUCER, NSM_SITE_STAGE_EMPTY)) return false;
        const uint32_t fb = R.bar(&R.ctrl->full[rp.stage]);
        ptx::mbar_arrive_expect_tx(fb, kSlot);
        const uint32_t slot = R.ring + static_cast<uint32_t>(rp.stage * kSlot);
        // the second panel may start past the matrix: it reads zeros
        const int x0 = c * kChunk, x1 = x0 + 64;
        if (bounds_ok(x0 >= 0 && x0 < job.n && (x0 & 7) == 0 && job.b >= 0, R.status, NSM_KERNEL_SMALL,
                      NSM_ROLE_PRODUCER, NSM_SITE_TMA_X_LOAD)) {
          ptx::tma_load_3d(slot, map, fb, x0, 0, job.b);
        }
        if (bounds_ok(x1 >= 0 && (x1 & 7) == 0 && job.b >= 0, R.status, NSM_KERNEL_SMALL, NSM_ROLE_PRODUCER,
                      NSM_SITE_TMA_X_LOAD)) {
          ptx::tma_load_3d(slot + kPanel, map, fb, x1, 0, job.b);
        }
        fill_parity[rp.stage] = static_cast<int>(rp.phase);
        rp.advance();
      }
    }
  }
  return true;
}

// ------------------------------------------------------------------ MMA issuer
template <bool FP16>
__device__ bool issue(const Roles& R, uint32_t tmem, const SmallJob* __restrict__ jobs, int njobs,
                      const SmallOp* __restrict__ ops, int nops) {
  const uint32_t id_sq = ptx::idesc_f16(128, 128, !FP16, false);
  const uint32_t id_pass = ptx::idesc_f16(128, kChunk, !FP16, true);
  RingPos rp;
  uint32_t acc_cnt = 0, sq_cnt = 0, xs = 0;
  uint32_t hand[2] = {0u, 0u};
  // m x m accumulator complete: hand it to the epilogue and wait until it is drained and
  // the rounded result is in shared memory
  auto finish_square = [&]() -> bool {
    ptx::mma_commit(R.bar(&R.ctrl->sq_full));
    if (!R.wait(&R.ctrl->sq_done, sq_cnt & 1u, NSM_ROLE_MMA, NSM_SITE_SQUARE_DONE)) return false;
    ++sq_cnt;
    ptx::tc_fence_after();
    return true;
  };
  // X' X'^T += chunk of X' in shared-memory slot `slot`
  auto accumulate_panel = [&](int c, uint32_t slot) -> bool {
    if (!R.wait(&R.ctrl->xt_full[slot], hand[slot] & 1u, NSM_ROLE_MMA, NSM_SITE_XT_FULL)) return false;
    ptx::tc_fence_after();
    const uint32_t base = R.xt + slot * kSlot;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      const uint64_t d = square_desc(base, kk);
      ptx::mma_f16(tmem, d, d, id_sq, (c | kk) != 0 ? 1u : 0u);
    }
    ptx::mma_commit(R.bar(&R.ctrl->xt_empty[slot]));
    ++hand[slot];
    return true;
  };
  for (int j = blockIdx.x; j < njobs; j += gridDim.x) {
    const SmallJob job = jobs[j];
    const int nck = (job.n + kChunk - 1) / kChunk;
    for (int o = 0; o < nops; ++o) {
      const SmallOp op = ops[o];
      if (op.kind == kSmallGram) {
        for (int c = 0; c < nck; ++c) {
          if (!R.wait(&R.ctrl->full[rp.stage], rp.phase, NSM_ROLE_MMA, NSM_SITE_STAGE_FULL)) return false;
          ptx::tc_fence_after();
          const uint32_t base = R.ring + static_cast<uint32_t>(rp.stage * kSlot);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint64_t d = square_desc(base, kk);
            ptx::mma_f16(tmem, d, d, id_sq, (c | kk) != 0 ? 1u : 0u);
          }
          ptx::mma_commit(R.bar(&R.ctrl->empty[rp.stage]));
          rp.advance();
        }
        if (!finish_square()) return false;
      } else if (op.kind == kSmallSquare) {
        const uint32_t a = R.square(op.a), b = R.square(op.b);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          ptx::mma_f16(tmem, square_desc(a, kk), square_desc(b, kk), id_sq, kk != 0 ? 1u : 0u);
        }
        if (!finish_square()) return false;
      } else {
        const uint32_t a = R.square(op.a);
        const uint32_t xs0 = xs;
        for (int c = 0; c < nck; ++c) {
          const uint32_t acc = acc_cnt & 1u;
          if (!R.wait(&R.ctrl->acc_empty[acc], ((acc_cnt >> 1) & 1u) ^ 1u, NSM_ROLE_MMA, NSM_SITE_ACC_EMPTY)) return false;
          ptx::tc_fence_after();
          if (!R.wait(&R.ctrl->full[rp.stage], rp.phase, NSM_ROLE_MMA, NSM_SITE_STAGE_FULL)) return false;
          ptx::tc_fence_after();
          // B = the chunk read K x N (N contiguous): two 64-column blocks kPanel apart
          const uint32_t chunk = R.ring + static_cast<uint32_t>(rp.stage * kSlot);
          const uint32_t d_tmem = tmem + 128u + static_cast<uint32_t>(kChunk) * acc;
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            ptx::mma_f16(d_tmem, square_desc(a, kk), ptx::smem_desc_sw128(chunk + kk * 2048, kPanel, 1024),
                         id_pass, kk != 0 ? 1u : 0u);
          }
          // with beta != 0 the epilogue reads the chunk too and releases it itself
          if (op.beta == 0.f) ptx::mma_commit(R.bar(&R.ctrl->empty[rp.stage]));
          ptx::mma_commit(R.bar(&R.ctrl->acc_full[acc]));
          ++acc_cnt;
          rp.advance();
          if (op.accumulate && c > 0) {
            if (!accumulate_panel(c - 1, (xs0 + c - 1) & 1u)) return false;
          }
        }
        if (op.accumulate) {
          if (!accumulate_panel(nck - 1, (xs0 + nck - 1) & 1u)) return false;
          if (!finish_square()) return false;
        }
        xs += static_cast<uint32_t>(nck);
      }
    }
  }
  return true;
}

// ------------------------------------------------------------------ epilogue (warps 2..5)
template <bool FP16>
struct Epilogue {
  using E = Store<FP16>;
  using T = typename E::T;
  const Roles& R;
  uint32_t t_lane;  // TMEM address of this warp's lane quarter, column 0
  int row;          // the accumulator row (= TMEM lane) this thread drains
  int lane;
  bool leader;      // first epilogue thread: issues the TMA stores
  uint32_t sq_cnt = 0;

  __device__ Epilogue(const Roles& r, uint32_t tmem, int warp, int ln)
      : R(r), lane(ln), leader(warp == 2 && ln == 0) {
    const int quarter = warp & 3;
    row = quarter * 32 + ln;
    t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
  }

  // Every epilogue thread waits; all give up together if any of them timed out.
  __device__ bool wait_all(uint64_t* b, uint32_t parity, int site) {
    const bool ok = R.wait(b, parity, NSM_ROLE_EPILOGUE, site);
    return ptx::named_all(kEpiBar, kEpiThreads, ok);
  }

  // S[dst] = alpha acc + beta S[aux] + diag I (rows < m on the diagonal)
  __device__ bool square(int dst, int aux, float alpha, float beta, float diag, int m) {
    if (!wait_all(&R.ctrl->sq_full, sq_cnt & 1u, NSM_SITE_SQUARE_FULL)) return false;
    ++sq_cnt;
    ptx::tc_fence_after();
    const uint32_t d = R.square(dst);
    const uint32_t x = aux >= 0 ? R.square(aux) : 0u;
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      uint32_t r[32];
      ptx::tmem_ld_32x32b_x32(t_lane + static_cast<uint32_t>(q * 32), r);
      ptx::tmem_ld_wait();
      float v[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) v[j] = alpha * __uint_as_float(r[j]);
      if (aux >= 0) {
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const int u = q * 4 + w;  // 16-byte unit of the row, 0..15
          const uint4 pk = *reinterpret_cast<const uint4*>(
              __cvta_shared_to_generic(x + (u >> 3) * kPanel + sw(row, u & 7)));
          const T* e = reinterpret_cast<const T*>(&pk);
#pragma unroll
          for (int k = 0; k < 8; ++k) v[w * 8 + k] += beta * E::to_f(e[k]);
        }
      }
      if (diag != 0.f && row < m) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          if (q * 32 + j == row) v[j] += diag;
        }
      }
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int u = q * 4 + w;
        uint4 pk;
        T* e = reinterpret_cast<T*>(&pk);
#pragma unroll
        for (int k = 0; k < 8; ++k) e[k] = E::from_f(v[w * 8 + k]);
        *reinterpret_cast<uint4*>(__cvta_shared_to_generic(d + (u >> 3) * kPanel + sw(row, u & 7))) = pk;
      }
    }
    ptx::tc_fence_before();
    ptx::fence_proxy_async_smem();  // the tensor cores read S[dst] next
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(R.bar(&R.ctrl->sq_done));
    return true;
  }
};

template <bool FP16>
__device__ bool drain(Epilogue<FP16>& ep, const SmallJob* __restrict__ jobs, int njobs,
                      const SmallOp* __restrict__ ops, int nops) {
  using E = Store<FP16>;
  using T = typename E::T;
  const Roles& R = ep.R;
  RingPos rp;
  uint32_t acc_cnt = 0, xs = 0;
  uint32_t hand[2] = {0u, 0u};
  int pend[2] = {-1, -1};  // parity of the MMA's outstanding read of each X' slot
  for (int j = blockIdx.x; j < njobs; j += gridDim.x) {
    const SmallJob job = jobs[j];
    const int nck = (job.n + kChunk - 1) / kChunk;
    for (int o = 0; o < nops; ++o) {
      const SmallOp op = ops[o];
      // an operation on the stored input (U 2^k) multiplies by s 2^-k, squared for X X^T
      const float f = op.in_pow == 0 ? 1.f : (op.in_pow == 2 ? job.in_scale[0] * job.in_scale[0] : job.in_scale[0]);
      if (op.kind == kSmallGram) {
        for (int c = 0; c < nck; ++c) rp.advance();
        if (!ep.square(op.dst, -1, f, 0.f, 0.f, job.m)) return false;
        continue;
      }
      if (op.kind == kSmallSquare) {
        if (!ep.square(op.dst, op.aux, op.alpha, op.beta, op.diag, job.m)) return false;
        continue;
      }
      const bool reads_x = op.beta != 0.f;
      const float alpha = op.alpha * f, beta = op.beta * f;
      const uint32_t xs0 = xs;
      for (int c = 0; c < nck; ++c) {
        const uint32_t acc = acc_cnt & 1u;
        bool ok = R.wait(&R.ctrl->acc_full[acc], (acc_cnt >> 1) & 1u, NSM_ROLE_EPILOGUE, NSM_SITE_ACC_FULL);
        if (ok && reads_x) ok = R.wait(&R.ctrl->full[rp.stage], rp.phase, NSM_ROLE_EPILOGUE, NSM_SITE_STAGE_FULL);
        if (!ptx::named_all(kEpiBar, kEpiThreads, ok)) return false;
        ptx::tc_fence_after();
        const int stage = rp.stage;
        const uint32_t chunk = R.ring + static_cast<uint32_t>(stage * kSlot);
        const uint32_t slot = (xs0 + static_cast<uint32_t>(c)) & 1u;
        {
          // the X' slot must be free: read by its store two chunks back and by the MMA
          if (ep.leader) ptx::bulk_wait_group_read<1>();
          bool free_ok = true;
          if (pend[slot] >= 0) {
            free_ok = R.wait(&R.ctrl->xt_empty[slot], static_cast<uint32_t>(pend[slot]), NSM_ROLE_EPILOGUE,
                             NSM_SITE_XT_EMPTY);
            pend[slot] = -1;
          }
          if (!ptx::named_all(kEpiBar, kEpiThreads, free_ok)) return false;
        }
        const uint32_t xt = R.xt + slot * kSlot;
        // the chunk's two 64-column halves, one panel each
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          float v[64];
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(
                ep.t_lane + 128u + static_cast<uint32_t>(kChunk) * acc + static_cast<uint32_t>(64 * h + 32 * q), r);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int k = 0; k < 32; ++k) v[q * 32 + k] = alpha * __uint_as_float(r[k]);
          }
          if (reads_x) {
            const uint32_t panel = chunk + static_cast<uint32_t>(h * kPanel);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              const uint4 pk = *reinterpret_cast<const uint4*>(__cvta_shared_to_generic(panel + sw(ep.row, u)));
              const T* e = reinterpret_cast<const T*>(&pk);
#pragma unroll
              for (int k = 0; k < 8; ++k) v[u * 8 + k] += beta * E::to_f(e[k]);
            }
          }
#pragma unroll
          for (int k = 0; k < 64; ++k) v[k] = E::to_f(E::from_f(v[k]));  // X' (or O) as stored
          const uint32_t dst = xt + static_cast<uint32_t>(h * kPanel);
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            uint4 pk;
            T* e = reinterpret_cast<T*>(&pk);
#pragma unroll
            for (int k = 0; k < 8; ++k) e[k] = E::from_f(v[u * 8 + k]);
            *reinterpret_cast<uint4*>(__cvta_shared_to_generic(dst + sw(ep.row, u))) = pk;
          }
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (ep.lane == 0) ptx::mbar_arrive(R.bar(&R.ctrl->acc_empty[acc]));
        ++acc_cnt;
        rp.advance();
        // X' (or O) chunk -> TMA stores (and to the MMA when accumulating)
        ptx::fence_proxy_async_smem();
        ptx::named_sync(kEpiBar, kEpiThreads);
        if (ep.leader) {
          if (reads_x) ptx::mbar_arrive(R.bar(&R.ctrl->empty[stage]));
          const int x0 = c * kChunk, x1 = x0 + 64;
          if (bounds_ok(x0 >= 0 && x0 < job.n && (x0 & 7) == 0 && job.b >= 0, R.status, NSM_KERNEL_SMALL,
                        NSM_ROLE_EPILOGUE, NSM_SITE_TMA_X_STORE)) {
            ptx::tma_store_3d(job.map_x[op.dst_x], xt, x0, 0, job.b);
          }
          if (x1 < job.n && bounds_ok((x1 & 7) == 0, R.status, NSM_KERNEL_SMALL, NSM_ROLE_EPILOGUE,
                                      NSM_SITE_TMA_X_STORE)) {
            ptx::tma_store_3d(job.map_x[op.dst_x], xt + kPanel, x1, 0, job.b);
          }
          ptx::bulk_commit_group();
        }
        if (op.accumulate) {
          if (ep.lane == 0) ptx::mbar_arrive(R.bar(&R.ctrl->xt_full[slot]));
          pend[slot] = static_cast<int>(hand[slot] & 1u);
          ++hand[slot];
        }
      }
      xs += static_cast<uint32_t>(nck);
      if (!op.final_pass && ep.leader) {
        // the next pass loads this X': every store must have landed
        ptx::bulk_wait_group<0>();
        ptx::fence_proxy_async_global();
        ptx::mbar_arrive(R.bar(&R.ctrl->stores_done));
      }
      if (op.accumulate) {
        if (!ep.square(op.dst, -1, 1.f, 0.f, 0.f, job.m)) return false;
      }
    }
  }
  return true;
}

template <bool FP16>
__global__ void __launch_bounds__(kThreads, 1)
    k_ns_small(const SmallJob* __restrict__ jobs, int njobs, const SmallOp* __restrict__ ops, int nops,
               int* status) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  Ctrl* ctrl = reinterpret_cast<Ctrl*>(smem + kCtrlOff);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  Roles R;
  R.ctrl = ctrl;
  R.squares = ptx::smem_u32(smem);
  R.ring = ptx::smem_u32(smem + kRingOff);
  R.xt = ptx::smem_u32(smem + kXtOff);
  R.status = status;
  R.abort_flag = &ctrl->abort;
  R.never_flag = &ctrl->never;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRing; ++s) {
      ptx::mbar_init(R.bar(&ctrl->full[s]), 1);
      ptx::mbar_init(R.bar(&ctrl->empty[s]), 1);
    }
    for (int a = 0; a < 2; ++a) {
      ptx::mbar_init(R.bar(&ctrl->acc_full[a]), 1);
      ptx::mbar_init(R.bar(&ctrl->acc_empty[a]), 4);
      ptx::mbar_init(R.bar(&ctrl->xt_full[a]), 4);
      ptx::mbar_init(R.bar(&ctrl->xt_empty[a]), 1);
    }
    ptx::mbar_init(R.bar(&ctrl->sq_full), 1);
    ptx::mbar_init(R.bar(&ctrl->sq_done), 4);
    ptx::mbar_init(R.bar(&ctrl->stores_done), 1);
    ptx::mbar_init(R.bar(&ctrl->drain), 1);
    ctrl->abort = 0;
    ctrl->never = 0;
    ptx::fence_mbarrier_init();
  }
  if (warp == 0) {
    ptx::tmem_alloc(ptx::smem_u32(&ctrl->tmem_base), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  // barriers and TMEM are set up; X comes from the previous kernel of the stream
  grid_dependency_sync();
  release_dependents();
  const uint32_t tmem = ctrl->tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      int fill_parity[kRing];
#pragma unroll
      for (int s = 0; s < kRing; ++s) fill_parity[s] = -1;
      if (!produce(R, jobs, njobs, ops, nops, fill_parity)) {
        R.give_up();
        // let every copy already issued land before the block can exit
        for (int s = 0; s < kRing; ++s) {
          if (fill_parity[s] >= 0) {
            ptx::mbar_wait_bounded(R.bar(&ctrl->full[s]), static_cast<uint32_t>(fill_parity[s]), R.never_flag,
                                   kWaitNs);
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      if (!issue<FP16>(R, tmem, jobs, njobs, ops, nops)) R.give_up();
      // no MMA may still write TMEM when the block frees it
      ptx::mma_commit(R.bar(&ctrl->drain));
      if (!ptx::mbar_wait_bounded(R.bar(&ctrl->drain), 0u, R.never_flag, kWaitNs)) {
        record_timeout(R.status, NSM_KERNEL_SMALL, NSM_ROLE_TEARDOWN, NSM_SITE_DRAIN);
        R.give_up();
      }
    }
    __syncwarp();
  } else {
    Epilogue<FP16> ep(R, tmem, warp, lane);
    drain<FP16>(ep, jobs, njobs, ops, nops);
    // stores still reading shared memory must finish before the block exits
    if (ep.leader) ptx::bulk_wait_group<0>();
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
}

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

template <bool FP16>
cudaError_t launch_typed(const SmallJob* jobs, int njobs, const SmallOp* ops, int nops, int num_sms,
                         cudaStream_t stream) {
  int* status = device_status_ptr();
  if (!status) return cudaErrorInvalidSymbol;
  static std::atomic<uint64_t> done{0};
  cudaError_t e = set_smem_once(k_ns_small<FP16>, kSmem, done);
  if (e != cudaSuccess) return e;
  const int grid = njobs < num_sms ? njobs : num_sms;
  if (grid <= 0) return cudaSuccess;
  if (const cudaError_t e_launch = launch_pdl(k_ns_small<FP16>, dim3(grid), dim3(kThreads), kSmem, stream, jobs, njobs, ops, nops, status)) return e_launch;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_ns_small(const SmallJob* jobs, int njobs, const SmallOp* ops, int nops, int fp16,
                            int num_sms, cudaStream_t stream) {
  if (nops <= 0 || nops > kSmallMaxOps) return cudaErrorInvalidValue;
  return fp16 ? launch_typed<true>(jobs, njobs, ops, nops, num_sms, stream)
              : launch_typed<false>(jobs, njobs, ops, nops, num_sms, stream);
}

}  // namespace nsm
