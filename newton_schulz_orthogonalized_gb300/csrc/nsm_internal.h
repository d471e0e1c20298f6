// Internal definitions shared by the host planner (nsm_api.cpp) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "nsmuon.h"

namespace nsm {

// Status word kernels write when a bounded wait expires (kDevTimeout in the low byte)
// or, in the checked build, when a bounds check fails (kDevBounds); then which kernel,
// which role inside it and which barrier or access site (NSM_KERNEL_*, NSM_ROLE_*,
// NSM_SITE_* of the public header).  Only the first record since the word was last read
// is kept.
constexpr int kDevOk = 0;
constexpr int kDevTimeout = 1;
constexpr int kDevBounds = 2;
__host__ __device__ constexpr int status_word(int kernel, int role, int site, int kind = kDevTimeout) {
  return kind | (kernel << 8) | (role << 16) | (site << 24);
}

// The checked build (compiled with NSM_CHECKED=1) tests every global access and TMA box of
// its kernels against the matrix it belongs to before making it.
#if defined(NSM_CHECKED) && NSM_CHECKED
constexpr bool kChecked = true;
#else
constexpr bool kChecked = false;
#endif

#ifdef __CUDACC__
__device__ __forceinline__ void record_timeout(int* status, int kernel, int role, int site) {
  atomicCAS(status, kDevOk, status_word(kernel, role, site));
}

// Whether an access may be made.  The regular build always says yes and the test
// compiles away; the checked build records a failed test (kDevBounds, kernel, role,
// site) and the caller skips the access.
__device__ __forceinline__ bool bounds_ok(bool ok, int* status, int kernel, int role, int site) {
  if constexpr (kChecked) {
    if (!ok) atomicCAS(status, kDevOk, status_word(kernel, role, site, kDevBounds));
    return ok;
  } else {
    return true;
  }
}
#endif

// Values of the process-wide launch options (NSM_OPT_* of the public header).
int option_value(int option);
// Whether the launches of the current library call use programmatic dependent launch
// (set per call from the NSM_OPT_PDL option and the size of the call's table).
bool pdl_for_launches();

// One matrix of a packed group, as the elementwise kernels see it.
struct MatInfo {
  int64_t off;        // element offset in the packed (natural, row-major) buffers
  int64_t slot;       // element offset of the matrix's slot in the class-layout buffers
  int64_t tile_begin; // prefix count of 64x64 natural tiles over the table
  int32_t rows, cols; // shape of the parameter
  int32_t m, n, ld;   // working shape (m = min, n = max) and row stride of the slot
  int32_t transposed; // rows > cols: the slot holds the transpose
  int32_t chunk_begin, nchunks;  // momentum/norm chunks of this matrix
  float scale;        // sqrt(max(1, rows/cols))
  int32_t flags;      // kMatVec
  int32_t cls_pos;    // position among the matrices in class order (class by class, batch index)
  int32_t pad;
};
// MatInfo::flags: rows % 8 == 0 && cols % 8 == 0 (16-byte vector paths usable)
constexpr int32_t kMatVec = 1;
static_assert(sizeof(MatInfo) == 72, "MatInfo layout");

// The normalised input X = s U of the chain is stored as U 2^k rounded once to the
// storage format, with a power-of-two k per matrix that puts its largest |U| in the
// format's normal range; the products that read it multiply by s 2^-k (the matrix's
// input factor, 'xs').  k is chosen so that the largest |U| 2^k lies in [2^11, 2^12); a
// stored value is accepted when it lies in [2^4, 2^15).
constexpr int kInTargetExp = 12;  // frexp exponent of max|U| 2^k after choosing k
constexpr int kInMinExp = 5;      // accepted: frexp exponent of max|U| 2^k in [5, 15]
constexpr int kInMaxExp = 15;
constexpr int kInExpClamp = 120;  // |k| at most this (2^k and 2^-k are normal floats)
// Partial sums (and maxima) the step's pass writes per 64 x 64 tile: one per warp of its
// 256-thread blocks, so that no block-wide barrier is needed to combine them.
constexpr int kTileParts = 8;

// e with x = f 2^e, f in [0.5, 1), of a positive finite float (subnormals count as 2^-126)
__host__ __device__ inline int in_frexp_exponent(float x) {
  uint32_t b;
  memcpy(&b, &x, sizeof b);
  const int biased = static_cast<int>((b >> 23) & 0xffu);
  return (biased == 0 ? 1 : biased) - 126;
}

__host__ __device__ inline int in_clamp_exp(int k) {
  return k < -kInExpClamp ? -kInExpClamp : (k > kInExpClamp ? kInExpClamp : k);
}

// The exponent of one matrix's stored input, from its largest |U| (max_abs), on the host
// and in k_scale_finalize alike.
struct InExponent {
  int k;      // U is (or is to be) stored as U 2^k
  int next;   // the hint for the next call on the table
  int store;  // 1: U must be stored with 2^k by the layout pass (0: what is stored stands)
};

// With a hint (the step), U was stored with 2^hint (clamped): that stands when
// max_abs 2^hint lies in [2^4, 2^15), and otherwise U is stored again with the exponent
// that puts max_abs 2^k in [2^11, 2^12), which is also the next hint.  Without a hint
// (the orthogonalisation) that exponent is the one used.  A matrix whose max_abs is 0,
// infinite or NaN yields no exponent: its hint (or 0) stands.
__host__ __device__ inline InExponent in_exponent(float max_abs, bool has_hint, int hint) {
  const bool has_max = max_abs > 0.f && max_abs <= 3.40282347e38f;
  const int e = has_max ? in_frexp_exponent(max_abs) : 0;
  InExponent r;
  if (has_hint) {
    const int used = in_clamp_exp(hint);
    const bool ok = !has_max || (e + used >= kInMinExp && e + used <= kInMaxExp);
    r.next = has_max ? in_clamp_exp(kInTargetExp - e) : used;
    r.k = ok ? used : r.next;
    r.store = ok ? 0 : 1;
  } else {
    r.k = has_max ? in_clamp_exp(kInTargetExp - e) : 0;
    r.next = r.k;
    r.store = 1;
  }
  return r;
}

// Elements of one momentum/norm chunk (256 threads x 8 vectors of 8).
constexpr int kChunk = 16384;
// Natural tiles moved between layouts are kTile x kTile.
constexpr int kTile = 64;

// One group of same-shape problems of a grouped GEMM launch:
//   out[b] = alpha * (A[b] . op(B[b])) + beta * aux[b] + diag * I     for b < count
// A[b] is M x K (K contiguous).  B[b] is N x K (K contiguous, "K-major") or K x N
// (N contiguous, "MN-major"), chosen per launch.  Output and aux are M x N with row
// strides ld_out / ld_aux and batch strides out_bstride / aux_bstride (elements).
// sym != 0: the output is known to be symmetric (M == N, aux symmetric); only the tiles
// in tile_list (packed mt << 16 | nt, tiles_per_mat of them) are computed, their upper
// triangle is stored and mirrored into the lower one.
// lean (2-SM kernel only, whose tiles are 256 x 256): symmetric m x m buffers stored as
// their upper 256 x 256 tiles.  kLeanOut: the output keeps only the tiles it computes
// (the diagonal tiles whole, no mirror of the others); kLeanA / kLeanB: the A / K-major B
// operand is such a buffer, so a 256-wide block below the diagonal (K block before the
// operand's own tile) is read from its mirror image above it, as an MN-major operand.
struct GemmGroup {
  const CUtensorMap* map_a;
  const CUtensorMap* map_b;
  void* out;
  const void* aux;
  const int32_t* tile_list;
  int64_t out_bstride;
  int64_t aux_bstride;
  int64_t tile_begin;
  int32_t ld_out, ld_aux;
  int32_t M, N, K;
  int32_t count;
  int32_t tiles_m, tiles_n;
  int32_t sym, tiles_per_mat;
  int32_t a_box, b_box;  // rows per TMA box of map_a / map_b (64, 128 or 256)
  const CUtensorMap* map_out;  // the output in 32 x 32 boxes with 64-byte swizzle (TMA stores);
                               // NULL when N is not a multiple of 8 (rows of whole 16-byte units)
  const CUtensorMap* map_b_narrow;  // B in 64-row boxes (K-major B; MN-major: map_b): the 2-SM
                                    // kernel's tiles with at most 128 columns in range
  int32_t lean;                     // kLeanOut | kLeanA | kLeanB (2-SM kernel only)
  int32_t in_pow;                   // 0, or 1 / 2: the product reads the chain's stored input
  const float* in_scale;            // in_pow != 0: input factor of problem b at in_scale[b];
                                    // the epilogue takes alpha, beta times in_scale[b]^in_pow
};
static_assert(sizeof(GemmGroup) == 144, "GemmGroup layout");
constexpr int32_t kLeanOut = 1;
constexpr int32_t kLeanA = 2;
constexpr int32_t kLeanB = 4;

struct GemmLaunch {
  const GemmGroup* groups;  // device array
  int32_t num_groups;
  int32_t b_mn_major;       // 1: B operand is K x N with N contiguous
  int32_t has_aux;
  int32_t fp16;             // 1: operands/outputs are fp16, else bf16
  int32_t pair;             // 1: 2-SM kernel on 256 x 256 tiles (groups laid out for it)
  int32_t narrow;           // 1 (pair only): some tile has at most 128 columns in range
  int64_t total_tiles;
  float alpha, beta, diag;
  double flops;             // flops the tensor cores execute (whole tiles)
  double canonical_flops;   // 2 M N K per problem, as if no tile were skipped
};

// ---- small-matrix kernel: the whole Newton-Schulz chain of one m <= 128 matrix per CTA

// Working shapes the small-matrix kernel takes: m (rows of the working matrix) at most this.
constexpr int kSmallMaxM = 128;

// One matrix for the small-matrix kernel: its class tensor maps of the two X buffers
// (128-row boxes), its batch index in the class and its MatInfo index.
struct SmallJob {
  const CUtensorMap* map_x[2];
  int32_t mat, b, m, n;
  const float* in_scale;  // the matrix's input factor (operations with in_pow read it)
};
static_assert(sizeof(SmallJob) == 40, "SmallJob layout");

// Operations of the small-matrix chain (every matrix of the launch runs the same list).
// S0..S2 are 128 x 128 matrices in shared memory, X0/X1 the class buffers in the workspace.
enum SmallOpKind : int32_t {
  kSmallGram = 0,    // S[dst] = X[src_x] X[src_x]^T
  kSmallSquare = 1,  // S[dst] = alpha S[a] S[b]^T + beta S[aux] + diag I
  kSmallPass = 2,    // X[dst_x] = alpha S[a] X[src_x] + beta X[src_x];
                     //   accumulate: also S[dst] = X[dst_x] X[dst_x]^T;  final: it is O
};
struct SmallOp {
  int32_t kind;
  int32_t a, b, dst, aux;  // shared-memory matrices; aux < 0: none
  int32_t src_x, dst_x;    // X buffers of Gram and pass operations
  int32_t accumulate, final_pass;
  float alpha, beta, diag;
  int32_t in_pow;          // reads the stored input: alpha, beta times the input factor^in_pow
};
static_assert(sizeof(SmallOp) == 52, "SmallOp layout");
constexpr int kSmallMaxOps = 96;

// ---- launchers (defined in the .cu files) ---------------------------------------

// Runs `ops` for every job; the final pass stores O into its X buffer.
cudaError_t launch_ns_small(const SmallJob* jobs, int njobs, const SmallOp* ops, int nops, int fp16,
                            int num_sms, cudaStream_t stream);

// Per-chunk sum of G^2 (partials[c]) and largest |G| (partials[total_chunks + c])
cudaError_t launch_grad_norm(const void* grads, const MatInfo* mats, int nmats, int total_chunks,
                             float* partials, cudaStream_t stream);
// M <- mu M + G and U = G + mu M (Nesterov) or M, stored as U 2^k (k = the matrix's
// hint) into the class layout, rounded once to bf16 (or fp16 when to_fp16); per tile t,
// kTileParts partial sums of U^2 (tparts[t kTileParts + w]) and largest |U| (the same
// index plus total_tiles kTileParts).  Clears *redo.
cudaError_t launch_momentum_class(const void* grads, float* momentum, int nesterov, float mu, void* dst,
                                  int to_fp16, const MatInfo* mats, int nmats, int64_t total_tiles,
                                  const int* hints, float* tparts, int* redo, cudaStream_t stream);
// Per matrix, from its partials (per chunk, or kTileParts per tile when by_tile; the
// maxima nparts entries after the sums): s = 1/(sqrt(sum) + eps) and the exponent k.
// With hints (the step): the stored U 2^hint is accepted or, with layout_scale = 2^k and
// *redo = 1, marked for the layout pass to store again (layout_scale 0 when accepted);
// hints receive the exponent for the next step.  Without: layout_scale = 2^k for the
// layout pass.  xs (matrix order) and xs_cls (class order) receive the input factor
// s 2^-k.
cudaError_t launch_scale_finalize(const MatInfo* mats, int nmats, const float* parts, int64_t nparts,
                                  int by_tile, int* hints, float* layout_scale, int* redo, float* xs,
                                  float* xs_cls, float eps, cudaStream_t stream);
// X = U 2^k (scales[i] = 2^k), U recomputed in fp32 from G and the updated M (or U = G),
// into the class layout, rounded once to bf16 (or fp16 when to_fp16).  redo != NULL: the
// step's second pass, which returns at once when *redo is 0 and otherwise leaves the
// matrices whose scale is 0 as they are.
cudaError_t launch_to_class(const void* grads, const float* momentum, int has_momentum, int nesterov,
                            float mu, void* dst, int to_fp16, const MatInfo* mats, int nmats,
                            int64_t total_tiles, const float* scales, const int* redo, cudaStream_t stream);
// class layout O -> p update in natural layout (and its bf16 copy when params_bf16 != NULL);
// o_scale (matrix order, may be NULL = 1): factor of each matrix's stored O
cudaError_t launch_apply(const void* o, int o_fp16, const float* o_scale, float* params, void* params_bf16,
                         const MatInfo* mats, int nmats, int64_t total_tiles, float lr, float wd,
                         cudaStream_t stream);
// class layout O -> natural bf16 copy (times o_scale, as for the apply)
cudaError_t launch_export(const void* o, int o_fp16, const float* o_scale, void* out, const MatInfo* mats,
                          int nmats, int64_t total_tiles, cudaStream_t stream);
cudaError_t launch_adamw(const void* grads, float* params, float* m, float* v,
                         int64_t numel, float lr, float beta1, float beta2, float eps,
                         float wd, float bc1, float bc2, cudaStream_t stream);
cudaError_t launch_gemm(const GemmLaunch& l, int num_sms, cudaStream_t stream);
// bytes from page-locked host memory (src_mapped: its device mapping) to device memory, by
// `ctas` CTAs of SM loads
cudaError_t launch_copy_h2d(void* dst, const void* src_mapped, size_t bytes, int ctas, cudaStream_t stream);

int* device_status_ptr();
// One CTA whose bounded wait expires after limit_ns and records kDevTimeout.
cudaError_t launch_status_selftest(uint64_t limit_ns, cudaStream_t stream);
// One thread that runs bounds_ok on an index past its range, making no access.
cudaError_t launch_bounds_selftest(cudaStream_t stream);

}  // namespace nsm
