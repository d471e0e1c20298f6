// C-ABI entry points of libnsmuon.so: argument validation, workspace layout, launch
// plans (tensor maps and grouped work lists) and the launch sequence of the Muon step.
//
// Sources ("DeepSpeed 集成 Muon 优化器实战" §use_muon参数打标, §核心算子,
// §混合优化器的参数组构造; "Z2 与 Z3 模式" §两种packed buffer生命周期).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <list>
#include <atomic>
#include <map>
#include <memory>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/nsmuon.h"
#include "nsm_internal.h"

namespace nsm {
namespace {

// Quintic coefficients of "DeepSpeed 集成 Muon 优化器实战" §核心算子.
constexpr float kA = 3.4445f;
constexpr float kB = -4.7750f;
constexpr float kC = 2.0315f;
constexpr float kNormEps = 1e-7f;
constexpr int kMaxSteps = 16;
// Gram form: R is re-anchored from the explicit iterate every 3 steps.  In fp16 storage
// that keeps the iteration as close to the exact one as every 2 steps does (about 2% on
// near-low-rank inputs; every 4: 2.5%, never: 10-47%), with 3 m^2 (n - m) fewer executed
// flops per five-step chain (symmetric products on half their tiles).
constexpr int kGramReanchor = 3;
constexpr int kMaxMatrices = 1 << 22;
constexpr int64_t kMaxDim = int64_t(1) << 30;
constexpr size_t kAlign = 1024;

thread_local std::string t_last_error;
thread_local int t_last_launches = 0;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return code;
}

int fail_cuda(cudaError_t e, const char* what) {
  return fail(NSM_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
int64_t align_up64(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------- layout

struct ShapeClass {
  int m, n;        // working shape, m <= n
  int ldn, ldm;    // row strides of the X slots and of the m x m buffers (multiples of 64)
  int count;
  int64_t x_base;  // element offset of the class in an X-layout buffer
  int64_t mm_base; // element offset of the class in an m x m buffer
};

struct Layout {
  int n = 0;
  int method = 0;
  int steps = 0;
  std::vector<ShapeClass> classes;
  std::vector<int> cls_of;
  std::vector<int> batch_of;
  std::vector<int64_t> slot;
  std::vector<int32_t> chunk_begin, nchunks;
  std::vector<int64_t> tile_begin;
  int64_t x_elems = 0, mm_elems = 0;
  int total_chunks = 0;
  int64_t total_tiles = 0;
  // partials: per chunk sums and maxima (2 x chunks) of the orthogonalisation's norm pass;
  // tparts: per tile sums and maxima (2 x kTileParts x tiles) of the step's pass; scales: the layout
  // pass's 2^k per matrix (0: nothing to store again); xs / xs_cls: the input factor
  // s 2^-k in matrix and class order; hints: the step's exponent per matrix, kept from one
  // call to the next
  size_t off_partials = 0, off_tparts = 0, off_scales = 0, off_xs = 0, off_xs_cls = 0, off_hints = 0;
  size_t off_redo = 0;  // one int: set when some matrix must be stored again
  size_t off_x[2] = {0, 0}, off_mm[4] = {0, 0, 0, 0};
  std::vector<int32_t> cls_pos;  // each matrix's position in class order
  std::vector<int32_t> cls_first;  // class order position of each class's first matrix
  int num_mm = 0;
  size_t bytes = 0;
};

int validate_shapes(const int32_t* shapes, int n) {
  if (!shapes) return fail(NSM_ERR_NULL, "shapes is NULL");
  if (n <= 0 || n > kMaxMatrices) return fail(NSM_ERR_SHAPE, "n = %d out of range", n);
  for (int i = 0; i < n; ++i) {
    const int64_t r = shapes[2 * i], c = shapes[2 * i + 1];
    if (r <= 0 || c <= 0) return fail(NSM_ERR_SHAPE, "matrix %d has shape %lldx%lld", i, (long long)r, (long long)c);
    if (r > kMaxDim || c > kMaxDim || r * c > (int64_t(1) << 40))
      return fail(NSM_ERR_SHAPE, "matrix %d is too large (%lldx%lld)", i, (long long)r, (long long)c);
  }
  return NSM_OK;
}

int validate_method(int method, int steps) {
  if (method != NSM_NS_STANDARD && method != NSM_NS_GRAM && method != NSM_NS_STANDARD_BF16)
    return fail(NSM_ERR_METHOD, "unknown ns_method %d (0 = standard, 1 = gram, 2 = standard_bf16)", method);
  if (steps < 0 || steps > kMaxSteps) return fail(NSM_ERR_METHOD, "ns_steps = %d not in [0, %d]", steps, kMaxSteps);
  return NSM_OK;
}

Layout make_layout(const int32_t* shapes, int n, int method, int steps) {
  Layout L;
  L.n = n;
  L.method = method;
  L.steps = steps;
  L.cls_of.resize(n);
  L.batch_of.resize(n);
  L.slot.resize(n);
  L.chunk_begin.resize(n);
  L.nchunks.resize(n);
  L.tile_begin.resize(n);
  std::map<std::pair<int, int>, int> index;
  for (int i = 0; i < n; ++i) {
    const int r = shapes[2 * i], c = shapes[2 * i + 1];
    const int m = std::min(r, c), nn = std::max(r, c);
    auto it = index.find({m, nn});
    int ci;
    if (it == index.end()) {
      ci = static_cast<int>(L.classes.size());
      index[{m, nn}] = ci;
      ShapeClass sc{};
      sc.m = m;
      sc.n = nn;
      sc.ldn = static_cast<int>(align_up64(nn, 64));
      sc.ldm = static_cast<int>(align_up64(m, 64));
      sc.count = 0;
      L.classes.push_back(sc);
    } else {
      ci = it->second;
    }
    L.cls_of[i] = ci;
    L.batch_of[i] = L.classes[ci].count++;
  }
  for (auto& sc : L.classes) {
    sc.x_base = L.x_elems;
    L.x_elems += int64_t(sc.count) * sc.m * sc.ldn;
    sc.mm_base = L.mm_elems;
    L.mm_elems += int64_t(sc.count) * sc.m * sc.ldm;
  }
  L.cls_first.resize(L.classes.size());
  for (size_t c = 0, pos = 0; c < L.classes.size(); ++c) {
    L.cls_first[c] = static_cast<int32_t>(pos);
    pos += size_t(L.classes[c].count);
  }
  L.cls_pos.resize(n);
  for (int i = 0; i < n; ++i) L.cls_pos[i] = L.cls_first[L.cls_of[i]] + L.batch_of[i];
  int64_t chunks = 0, tiles = 0;
  for (int i = 0; i < n; ++i) {
    const ShapeClass& sc = L.classes[L.cls_of[i]];
    L.slot[i] = sc.x_base + int64_t(L.batch_of[i]) * sc.m * sc.ldn;
    const int64_t len = int64_t(shapes[2 * i]) * shapes[2 * i + 1];
    L.chunk_begin[i] = static_cast<int32_t>(chunks);
    L.nchunks[i] = static_cast<int32_t>((len + kChunk - 1) / kChunk);
    chunks += L.nchunks[i];
    L.tile_begin[i] = tiles;
    tiles += int64_t((shapes[2 * i] + kTile - 1) / kTile) * ((shapes[2 * i + 1] + kTile - 1) / kTile);
  }
  L.total_chunks = static_cast<int>(std::min<int64_t>(chunks, INT32_MAX));
  L.total_tiles = tiles;
  L.num_mm = method == NSM_NS_GRAM ? 4 : 2;
  size_t off = 0;
  L.off_hints = off;  // first, so that the same table finds them at the same place
  off = align_up(off + size_t(n) * 4, kAlign);
  L.off_partials = off;
  off = align_up(off + size_t(chunks) * 8, kAlign);
  L.off_tparts = off;
  off = align_up(off + size_t(tiles) * 8 * kTileParts, kAlign);
  L.off_redo = off;
  off = align_up(off + 4, kAlign);
  L.off_scales = off;
  off = align_up(off + size_t(n) * 4, kAlign);
  L.off_xs = off;
  off = align_up(off + size_t(n) * 4, kAlign);
  L.off_xs_cls = off;
  off = align_up(off + size_t(n) * 4, kAlign);
  for (int k = 0; k < 2; ++k) {
    L.off_x[k] = off;
    off = align_up(off + size_t(L.x_elems) * 2, kAlign);
  }
  for (int k = 0; k < L.num_mm; ++k) {
    L.off_mm[k] = off;
    off = align_up(off + size_t(L.mm_elems) * 2, kAlign);
  }
  L.bytes = off;
  return L;
}

// ---------------------------------------------------------------- tensor maps

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                    const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                    const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                    CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      fn = reinterpret_cast<EncodeTiledFn>(p);
    }
  });
  return fn;
}

// 3D map over `count` back-to-back row-major matrices of rows x inner (row stride ld),
// box 64 x box_rows x 1, 128-byte swizzle, zero fill outside the matrix.
// 3D map {inner, rows, count} of 16-bit elements.  Load maps take 64-wide boxes of
// box_rows rows with 128-byte swizzle; store maps (store = true) 32 x 32 boxes with
// 64-byte swizzle.
int encode_map(CUtensorMap* map, void* base, bool fp16, int inner, int rows, int ld, int count,
               const char* ws_begin, const char* ws_end, int box_rows = 64, bool store = false) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return fail(NSM_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  const size_t row_bytes = size_t(ld) * 2;
  const size_t mat_bytes = size_t(rows) * row_bytes;
  const char* first = static_cast<const char*>(base);
  const char* last = first + size_t(count - 1) * mat_bytes + size_t(rows - 1) * row_bytes + size_t(inner) * 2;
  if (ws_begin && (first < ws_begin || last > ws_end))
    return fail(NSM_ERR_WORKSPACE, "internal: tensor map exceeds the workspace");
  cuuint64_t dims[3] = {cuuint64_t(inner), cuuint64_t(rows), cuuint64_t(count)};
  cuuint64_t strides[2] = {cuuint64_t(row_bytes), cuuint64_t(mat_bytes)};
  cuuint32_t box[3] = {store ? 32u : 64u, store ? 32u : static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, fp16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base,
                  dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  store ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(NSM_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", int(r));
  return NSM_OK;
}

// ---------------------------------------------------------------- plans

// Buffers the chain reads/writes, per class: X0, X1 (X layout) and MM0..MM3 (m x m).
enum Buf { X0 = 0, X1 = 1, MM0 = 2 };

struct Plan {
  Layout L;
  int device = 0;
  char* ws = nullptr;
  void* dmeta = nullptr;
  MatInfo* d_mats = nullptr;
  std::vector<GemmLaunch> launches;
  int64_t elems = 0;      // elements of the table (sum of rows x cols)
  int final_buf = X0;     // buffer holding O after the chain
  bool final_is_input = false;  // no step: O is the stored input (U 2^k, factor s 2^-k)
  bool final_fp16 = false;
  bool x_fp16 = false;
  bool owns_meta = true;  // false when the metadata lives in memory the plan does not own
  // matrices with m <= kSmallMaxM run their whole chain in the small-matrix kernel
  const SmallJob* d_small_jobs = nullptr;
  const SmallOp* d_small_ops = nullptr;
  int n_small_jobs = 0;
  int n_small_ops = 0;
  double small_bytes = 0;  // HBM bytes the small-matrix kernel must move (its roofline)
  bool lean = false;       // symmetric iterates stored as their upper 256 x 256 tiles
  ~Plan() {
    if (dmeta && owns_meta) cudaFree(dmeta);
  }
};

// Process-wide launch options (nsm_set_option).  The 2-SM kernel is used where it pays,
// matrices with m <= 128 run in the small-matrix kernel and symmetric iterates are stored
// as their upper tiles where the chain allows it, unless an option says otherwise (for
// comparisons); programmatic dependent launch is automatic (on for small tables).
std::atomic<int> g_opt_pair{1}, g_opt_small{1}, g_opt_pdl{2}, g_opt_lean{1};

// Programmatic dependent launch for the current call: on (1), off (0), or, in the auto
// mode (2), on for tables of at most kPdlAutoElems elements, where each kernel is short
// and the launch latency it hides is a visible share of the step.
constexpr int64_t kPdlAutoElems = int64_t(1) << 25;
thread_local bool t_pdl = false;

struct PdlScope {
  explicit PdlScope(int64_t elems) {
    const int o = g_opt_pdl.load();
    t_pdl = o == 1 || (o == 2 && elems <= kPdlAutoElems);
  }
  ~PdlScope() { t_pdl = false; }
};

bool pair_kernels_enabled() { return g_opt_pair.load() != 0; }
bool small_kernel_enabled() { return g_opt_small.load() != 0; }
bool lean_storage_enabled() { return g_opt_lean.load() != 0; }

// Flops of one matrix's Newton-Schulz chain (2 m n k per product, as if no tile were
// skipped): standard 4 m^2 n + 2 m^3 per step; gram counts its m x n products (X X^T,
// Q X) and m x m products step by step, with re-anchoring.
int64_t chain_flops(int method, int steps, int64_t m, int64_t n) {
  if (method == NSM_NS_GRAM) {
    int64_t wide = steps > 0 ? 1 : 0, cubes = 0;
    bool q_identity = true;
    for (int k = 1; k <= steps; ++k) {
      cubes += q_identity ? 1 : 2;
      q_identity = false;
      if (k < steps) {
        if (k % kGramReanchor == 0) {
          wide += 2;
          q_identity = true;
        } else {
          cubes += 2;
        }
      }
    }
    if (steps > 0 && !q_identity) wide += 1;
    return 2 * wide * m * m * n + 2 * cubes * m * m * m;
  }
  return int64_t(steps) * (4 * m * m * n + 2 * m * m * m);
}

// The chain of one matrix as the small-matrix kernel runs it: the products and storage
// points of the grouped stages, with X X^T of each new iterate accumulated by the pass
// that forms it.  S0..S2 are the kernel's shared-memory matrices.  Returns the X buffer
// that receives O (the one the grouped stages end in).
int small_schedule(int method, int steps, std::vector<SmallOp>& ops) {
  auto make = [](int kind) {
    SmallOp o{};
    o.kind = kind;
    o.aux = -1;
    o.alpha = 1.f;
    return o;
  };
  if (method == NSM_NS_GRAM) {
    int xb = X0;
    bool xb_input = true;  // X[xb] is still the stored input
    int q = -1;  // shared-memory matrix holding Q; -1 = identity
    SmallOp g = make(kSmallGram);  // R = X X^T in S0
    g.src_x = xb;
    g.dst = 0;
    g.in_pow = 2;
    ops.push_back(g);
    for (int k = 1; k <= steps; ++k) {
      const int h = q == 1 ? 2 : 1;
      SmallOp hs = make(kSmallSquare);  // H = a I + b R + c R R
      hs.a = 0;
      hs.b = 0;
      hs.dst = h;
      hs.aux = 0;
      hs.alpha = kC;
      hs.beta = kB;
      hs.diag = kA;
      ops.push_back(hs);
      if (q < 0) {
        q = h;  // Q = H
      } else {
        SmallOp qs = make(kSmallSquare);  // Q = H Q, in place
        qs.a = h;
        qs.b = q;
        qs.dst = q;
        ops.push_back(qs);
      }
      if (k < steps) {
        if (k % kGramReanchor == 0) {
          const int xn = xb == X0 ? X1 : X0;
          SmallOp ps = make(kSmallPass);  // X = Q X, and R = X X^T on the way
          ps.a = q;
          ps.src_x = xb;
          ps.dst_x = xn;
          ps.accumulate = 1;
          ps.dst = 0;
          ps.in_pow = xb_input ? 1 : 0;
          ops.push_back(ps);
          xb = xn;
          xb_input = false;
          q = -1;
        } else {
          SmallOp ts = make(kSmallSquare);  // T = H R, in R's place
          ts.a = h;
          ts.b = 0;
          ts.dst = 0;
          ops.push_back(ts);
          SmallOp rs = make(kSmallSquare);  // R = T H
          rs.a = 0;
          rs.b = h;
          rs.dst = 0;
          ops.push_back(rs);
        }
      }
    }
    const int xn = xb == X0 ? X1 : X0;
    SmallOp fs = make(kSmallPass);  // O = Q X
    fs.a = q;
    fs.src_x = xb;
    fs.dst_x = xn;
    fs.final_pass = 1;
    fs.in_pow = xb_input ? 1 : 0;
    ops.push_back(fs);
    return xn;
  }
  SmallOp g = make(kSmallGram);  // A = X X^T in S0
  g.src_x = X0;
  g.dst = 0;
  g.in_pow = 2;
  ops.push_back(g);
  for (int k = 0; k < steps; ++k) {
    const int src = (k % 2 == 0) ? X0 : X1, dst = (k % 2 == 0) ? X1 : X0;
    SmallOp bs = make(kSmallSquare);  // B = b A + c A A in S1
    bs.a = 0;
    bs.b = 0;
    bs.dst = 1;
    bs.aux = 0;
    bs.alpha = kC;
    bs.beta = kB;
    ops.push_back(bs);
    SmallOp ps = make(kSmallPass);  // X' = a X + B X (and A = X' X'^T unless last)
    ps.a = 1;
    ps.src_x = src;
    ps.dst_x = dst;
    ps.beta = kA;
    ps.in_pow = k == 0 ? 1 : 0;
    if (k + 1 < steps) {
      ps.accumulate = 1;
      ps.dst = 0;
    } else {
      ps.final_pass = 1;
    }
    ops.push_back(ps);
  }
  return steps % 2 == 0 ? X0 : X1;
}

// Device memory a caller provides for a plan's metadata instead of a fresh allocation.
struct MetaSink {
  char* dptr;
  size_t capacity;
  cudaStream_t stream;
};

struct StageSpec {
  int a_buf, b_buf, out_buf, aux_buf;  // aux_buf < 0: none
  bool b_mn;                           // B operand is the X slot read K x N
  bool k_is_n;                         // K = n (X X^T); otherwise K = m
  bool n_is_n;                         // N = n (B X, Q X); otherwise N = m
  float alpha, beta, diag;
  bool sym;                            // output symmetric: upper-triangle tiles + mirror
  int in_pow;                          // reads the stored input: 1, or 2 for X X^T; else 0
};

// Tiles (packed mt << 16 | nt) of an m x m output that touch its upper triangle, for
// tiles of tile_m rows and 256 columns, in the engine's panel raster (panels of 2 column
// tiles, rows inside a panel).
std::vector<int32_t> upper_tiles(int m, int tile_m = 128) {
  std::vector<int32_t> t;
  const int tm = (m + tile_m - 1) / tile_m, tn = (m + 255) / 256;
  constexpr int kPanel = 2;
  for (int p0 = 0; p0 < tn; p0 += kPanel)
    for (int mt = 0; mt < tm; ++mt)
      for (int nt = p0; nt < std::min(p0 + kPanel, tn); ++nt)
        if (std::min(nt * 256 + 255, m - 1) >= mt * tile_m) t.push_back((mt << 16) | nt);
  return t;
}

// Flops the tensor cores execute for the listed tiles of an m x m x K product.
double tile_flops(const std::vector<int32_t>& tiles, int m, int K, int tile_m = 128) {
  double f = 0;
  for (int32_t p : tiles) {
    const int mt = p >> 16, nt = p & 0xffff;
    f += 2.0 * K * std::min(tile_m, m - mt * tile_m) * std::min(256, m - nt * 256);
  }
  return f;
}

// The 2-SM kernel pays off when most of a launch's work has at least 256 rows per tile;
// matrices with fewer rows would leave half of each pair idle.
bool prefer_pair(const std::vector<std::pair<int, double>>& rows_and_flops) {
  double big = 0, all = 0;
  for (const auto& rf : rows_and_flops) {
    all += rf.second;
    if (rf.first >= 256) big += rf.second;
  }
  return all > 0 && big >= 0.75 * all;
}

int build_plan(Plan& P, const int32_t* shapes, const int64_t* offsets, int n, int method, int steps,
               void* ws, size_t ws_bytes, const MetaSink* sink = nullptr) {
  P.L = make_layout(shapes, n, method, steps);
  const Layout& L = P.L;
  const bool use_pair_kernels = pair_kernels_enabled();
  for (int i = 0; i < n; ++i) P.elems += int64_t(shapes[2 * i]) * shapes[2 * i + 1];
  P.ws = static_cast<char*>(ws);
  P.x_fp16 = method != NSM_NS_STANDARD_BF16;
  P.final_is_input = steps == 0;
  const int nclass = static_cast<int>(L.classes.size());
  const int nbuf = 2 + L.num_mm;
  auto buf_base = [&](int b, int c) -> char* {
    const ShapeClass& sc = L.classes[c];
    if (b < MM0) return P.ws + L.off_x[b] + size_t(sc.x_base) * 2;
    return P.ws + L.off_mm[b - MM0] + size_t(sc.mm_base) * 2;
  };

  // Launch list of the chain.
  std::vector<StageSpec> stages;
  if (method == NSM_NS_STANDARD || method == NSM_NS_STANDARD_BF16) {
    for (int k = 0; k < steps; ++k) {
      const int src = (k % 2 == 0) ? X0 : X1, dst = (k % 2 == 0) ? X1 : X0;
      const int first = k == 0 ? 1 : 0;  // the first step reads the stored input
      stages.push_back({src, src, MM0, -1, false, true, false, 1.f, 0.f, 0.f, true, 2 * first});   // A = X X^T
      stages.push_back({MM0, MM0, MM0 + 1, MM0, false, false, false, kC, kB, 0.f, true, 0});        // B = bA + cAA
      stages.push_back({MM0 + 1, src, dst, src, true, false, true, 1.f, kA, 0.f, false, first});     // X' = aX + BX
    }
    P.final_buf = (steps % 2 == 0) ? X0 : X1;
    P.final_fp16 = P.x_fp16;
  } else {
    // Gram form ("DeepSpeed 集成 Muon 优化器实战" §核心算子): iterate on R = X X^T in fp16,
    // accumulate Q, re-anchor (X <- Q X, R <- X X^T, Q <- I) every kGramReanchor steps.
    // Four m x m buffers suffice: R, Q, H and one temporary (T or the new Q).
    int xb = X0;      // buffer holding the current anchor X
    int rR = MM0;     // R
    int q = -1;       // Q, -1 = identity
    std::vector<int> freeb = {MM0 + 1, MM0 + 2, MM0 + 3};
    auto pop = [&]() {
      const int b = freeb.front();
      freeb.erase(freeb.begin());
      return b;
    };
    auto push = [&](int b) { freeb.push_back(b); };
    bool xb_input = true;  // the anchor X is still the stored input
    if (steps > 0) stages.push_back({xb, xb, rR, -1, false, true, false, 1.f, 0.f, 0.f, true, 2});    // R = X X^T
    for (int k = 1; k <= steps; ++k) {
      const int h = pop();
      stages.push_back({rR, rR, h, rR, false, false, false, kC, kB, kA, true});                        // H
      bool h_is_q = false;
      if (q < 0) {
        q = h;                                                                                    // Q = H
        h_is_q = true;
      } else {
        const int qn = pop();
        stages.push_back({h, q, qn, -1, false, false, false, 1.f, 0.f, 0.f, true});                    // Q' = H Q
        push(q);
        q = qn;
      }
      if (k < steps) {
        if (k % kGramReanchor == 0) {
          const int xn = (xb == X0) ? X1 : X0;
          stages.push_back({q, xb, xn, -1, true, false, true, 1.f, 0.f, 0.f, false, xb_input ? 1 : 0});  // X = Q X
          xb = xn;
          xb_input = false;
          stages.push_back({xb, xb, rR, -1, false, true, false, 1.f, 0.f, 0.f, true, 0});              // R = X X^T
          push(q);  // H is Q here or already released below
          if (!h_is_q) push(h);
          q = -1;
          continue;
        }
        const int t = pop();
        stages.push_back({h, rR, t, -1, false, false, false, 1.f, 0.f, 0.f, true});                    // T = H R
        stages.push_back({t, h, rR, -1, false, false, false, 1.f, 0.f, 0.f, true});                    // R = T H
        push(t);
      }
      if (!h_is_q) push(h);
    }
    if (q >= 0) {
      const int xn = (xb == X0) ? X1 : X0;
      stages.push_back({q, xb, xn, -1, true, false, true, 1.f, 0.f, 0.f, false, xb_input ? 1 : 0});    // O = Q X
      P.final_buf = xn;
    } else {
      P.final_buf = xb;
    }
    P.final_fp16 = true;
  }

  // Upper-triangle tile lists of the m x m products, one per class and tile height
  // (index 0: 128-row tiles of the 1-CTA kernel, 1: 256-row tiles of the pair kernel).
  std::vector<std::vector<int32_t>> class_tiles[2];
  std::vector<size_t> tiles_off[2];
  size_t tile_ints = 0;
  for (int k = 0; k < 2; ++k) {
    class_tiles[k].resize(nclass);
    tiles_off[k].resize(nclass);
    for (int c = 0; c < nclass; ++c) {
      class_tiles[k][c] = upper_tiles(L.classes[c].m, k ? 256 : 128);
      tiles_off[k][c] = tile_ints;
      tile_ints += class_tiles[k][c].size();
    }
  }

  // Classes whose whole chain runs in the small-matrix kernel; the grouped launches take
  // the others.
  std::vector<char> small(nclass, 0);
  std::vector<int> big;
  for (int c = 0; c < nclass; ++c) {
    small[c] = steps > 0 && small_kernel_enabled() && L.classes[c].m <= kSmallMaxM;
    if (!small[c]) big.push_back(c);
  }
  std::vector<SmallOp> small_ops;
  std::vector<int> small_mats;
  for (int i = 0; i < n; ++i) {
    if (small[L.cls_of[i]]) small_mats.push_back(i);
  }
  if (!small_mats.empty()) {
    const int final_x = small_schedule(method, steps, small_ops);
    if (final_x != P.final_buf || small_ops.size() > size_t(kSmallMaxOps))
      return fail(NSM_ERR_METHOD, "small-matrix schedule does not fit (%zu operations)", small_ops.size());
    // heaviest first, for the persistent CTAs' balance
    std::stable_sort(small_mats.begin(), small_mats.end(), [&](int x, int y) {
      return int64_t(shapes[2 * x]) * shapes[2 * x + 1] > int64_t(shapes[2 * y]) * shapes[2 * y + 1];
    });
    // every Gram and pass operation reads X once, every pass writes X' (or O) once
    int x_reads = 0, x_writes = 0;
    for (const SmallOp& o : small_ops) {
      if (o.kind != kSmallSquare) ++x_reads;
      if (o.kind == kSmallPass) ++x_writes;
    }
    for (int i : small_mats) {
      const ShapeClass& sc = L.classes[L.cls_of[i]];
      P.small_bytes += 2.0 * double(sc.m) * double(sc.n) * (x_reads + x_writes);
    }
  }

  // Device metadata: MatInfo[n] | tensor maps [nclass][nbuf] | GemmGroup arrays | tile
  // lists | small-matrix jobs | small-matrix operations.
  const size_t mats_bytes = align_up(sizeof(MatInfo) * n, 128);
  const size_t maps_off = mats_bytes;
  constexpr int kBoxKinds = 4;  // load boxes of 64, 128, 256 rows; 32 x 32 store boxes
  const size_t maps_bytes = align_up(sizeof(CUtensorMap) * size_t(nclass) * nbuf * kBoxKinds, 128);
  const size_t groups_off = maps_off + maps_bytes;
  const size_t groups_bytes = align_up(sizeof(GemmGroup) * size_t(nclass) * stages.size(), 128);
  const size_t tiles_off_bytes = groups_off + groups_bytes;
  const size_t jobs_off = align_up(tiles_off_bytes + tile_ints * sizeof(int32_t), 128);
  const size_t ops_off = align_up(jobs_off + sizeof(SmallJob) * small_mats.size(), 128);
  const size_t total = ops_off + sizeof(SmallOp) * small_ops.size() + 128;
  std::vector<uint8_t> host(total, 0);

  MatInfo* hm = reinterpret_cast<MatInfo*>(host.data());
  for (int i = 0; i < n; ++i) {
    const ShapeClass& sc = L.classes[L.cls_of[i]];
    MatInfo mi{};
    mi.off = offsets ? offsets[i] : 0;
    mi.slot = L.slot[i];
    mi.tile_begin = L.tile_begin[i];
    mi.rows = shapes[2 * i];
    mi.cols = shapes[2 * i + 1];
    mi.m = sc.m;
    mi.n = sc.n;
    mi.ld = sc.ldn;
    mi.transposed = mi.rows > mi.cols ? 1 : 0;
    mi.chunk_begin = L.chunk_begin[i];
    mi.nchunks = L.nchunks[i];
    mi.scale = static_cast<float>(std::sqrt(std::max(1.0, double(mi.rows) / double(mi.cols))));
    mi.flags = (mi.rows % 8 == 0 && mi.cols % 8 == 0) ? kMatVec : 0;
    mi.cls_pos = L.cls_pos[i];
    hm[i] = mi;
  }

  cudaError_t e = cudaSuccess;
  if (sink) {
    if (total > sink->capacity)
      return fail(NSM_ERR_WORKSPACE, "plan metadata needs %zu bytes, %zu available", total, sink->capacity);
    P.dmeta = sink->dptr;
    P.owns_meta = false;
  } else {
    e = cudaMalloc(&P.dmeta, total);
    if (e != cudaSuccess) return fail_cuda(e, "cudaMalloc(plan metadata)");
  }
  char* dbase = static_cast<char*>(P.dmeta);
  P.d_mats = reinterpret_cast<MatInfo*>(dbase);

  const char* ws_begin = P.ws;
  const char* ws_end = P.ws + L.bytes;
  CUtensorMap* hmaps = reinterpret_cast<CUtensorMap*>(host.data() + maps_off);
  for (int c = 0; c < nclass; ++c) {
    const ShapeClass& sc = L.classes[c];
    for (int b = 0; b < nbuf; ++b) {
      for (int k = 0; k < kBoxKinds; ++k) {
        CUtensorMap* map = &hmaps[(size_t(c) * nbuf + b) * kBoxKinds + k];
        const int box = 64 << (k % 3);
        const bool store = k == 3;
        int rc;
        if (b < MM0)
          rc = encode_map(map, buf_base(b, c), P.x_fp16, sc.n, sc.m, sc.ldn, sc.count, ws_begin, ws_end, box, store);
        else
          rc = encode_map(map, buf_base(b, c), P.x_fp16, sc.m, sc.m, sc.ldm, sc.count, ws_begin, ws_end, box, store);
        if (rc != NSM_OK) return rc;
      }
    }
  }
  // map of buffer b of class c with load boxes of `box` rows, or its store map (box 0)
  auto dmap = [&](int c, int b, int box) {
    const int k = box == 0 ? 3 : (box >= 256 ? 2 : (box >= 128 ? 1 : 0));
    return reinterpret_cast<const CUtensorMap*>(dbase + maps_off) + (size_t(c) * nbuf + b) * kBoxKinds + k;
  };

  int32_t* htiles = reinterpret_cast<int32_t*>(host.data() + tiles_off_bytes);
  for (int k = 0; k < 2; ++k) {
    for (int c = 0; c < nclass; ++c) {
      std::copy(class_tiles[k][c].begin(), class_tiles[k][c].end(), htiles + tiles_off[k][c]);
    }
  }
  const int32_t* dtiles = reinterpret_cast<const int32_t*>(dbase + tiles_off_bytes);
  if (!small_mats.empty()) {
    SmallJob* hj = reinterpret_cast<SmallJob*>(host.data() + jobs_off);
    for (size_t k = 0; k < small_mats.size(); ++k) {
      const int i = small_mats[k];
      const int c = L.cls_of[i];
      SmallJob jb{};
      jb.map_x[0] = dmap(c, X0, 128);
      jb.map_x[1] = dmap(c, X1, 128);
      jb.mat = i;
      jb.b = L.batch_of[i];
      jb.m = L.classes[c].m;
      jb.n = L.classes[c].n;
      jb.in_scale = reinterpret_cast<const float*>(P.ws + L.off_xs) + i;
      hj[k] = jb;
    }
    std::copy(small_ops.begin(), small_ops.end(), reinterpret_cast<SmallOp*>(host.data() + ops_off));
    P.d_small_jobs = reinterpret_cast<const SmallJob*>(dbase + jobs_off);
    P.d_small_ops = reinterpret_cast<const SmallOp*>(dbase + ops_off);
    P.n_small_jobs = static_cast<int>(small_mats.size());
    P.n_small_ops = static_cast<int>(small_ops.size());
  }
  GemmGroup* hg = reinterpret_cast<GemmGroup*>(host.data() + groups_off);
  const int nbig = static_cast<int>(big.size());
  // The 2-SM kernel where most of a launch's work has at least 256 rows per tile.
  auto stage_pair = [&](const StageSpec& st) {
    std::vector<std::pair<int, double>> rows_and_flops;
    for (int c : big) {
      const ShapeClass& sc = L.classes[c];
      const double f = 2.0 * sc.count * double(sc.m) * (st.n_is_n ? sc.n : sc.m) * (st.k_is_n ? sc.n : sc.m);
      rows_and_flops.push_back({sc.m, f});
    }
    return use_pair_kernels && prefer_pair(rows_and_flops);
  };
  // Symmetric iterates stored as their upper 256 x 256 tiles: only where every launch of
  // the chain is on the 2-SM kernel (its tiles are 256 x 256; the 1-CTA kernel reads and
  // writes whole matrices).
  bool lean = lean_storage_enabled() && nbig > 0;
  for (const StageSpec& st : stages) lean = lean && stage_pair(st);
  P.lean = lean;
  for (size_t s = 0; s < stages.size() && nbig > 0; ++s) {
    const StageSpec& st = stages[s];
    // heaviest tiles (largest K) first
    std::vector<int> order = big;
    std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
      const int kx = st.k_is_n ? L.classes[x].n : L.classes[x].m;
      const int ky = st.k_is_n ? L.classes[y].n : L.classes[y].m;
      return kx > ky;
    });
    GemmGroup* gs = hg + s * nclass;
    int64_t tiles = 0;
    double flops = 0, canonical = 0;
    const bool pair = stage_pair(st);
    const int tile_m = pair ? 256 : 128;
    const int tk = pair ? 1 : 0;
    for (int j = 0; j < nbig; ++j) {
      const int c = order[j];
      const ShapeClass& sc = L.classes[c];
      GemmGroup g{};
      // the largest boxes each kernel can use: A halves and K-major B halves of 128 rows
      // (pair) or A 128 rows and K-major B 256 rows (1-CTA); MN-major B in 64 x 64 boxes
      g.a_box = 128;
      g.b_box = st.b_mn ? (pair ? 128 : 64) : (pair ? 128 : 256);
      g.map_a = dmap(c, st.a_buf, g.a_box);
      g.map_b = dmap(c, st.b_buf, g.b_box);
      g.map_b_narrow = st.b_mn ? g.map_b : dmap(c, st.b_buf, 64);
      const bool out_x = st.out_buf < MM0;
      g.out = buf_base(st.out_buf, c);
      // TMA stores write whole 16-byte units of a row: only for rows of a multiple of 8
      g.map_out = ((st.n_is_n ? sc.n : sc.m) % 8 == 0) ? dmap(c, st.out_buf, 0) : nullptr;
      g.ld_out = out_x ? sc.ldn : sc.ldm;
      g.out_bstride = int64_t(sc.m) * g.ld_out;
      if (st.aux_buf >= 0) {
        const bool aux_x = st.aux_buf < MM0;
        g.aux = buf_base(st.aux_buf, c);
        g.ld_aux = aux_x ? sc.ldn : sc.ldm;
        g.aux_bstride = int64_t(sc.m) * g.ld_aux;
      }
      if (st.in_pow) {
        g.in_pow = st.in_pow;
        g.in_scale = reinterpret_cast<const float*>(P.ws + L.off_xs_cls) + L.cls_first[c];
      }
      g.M = sc.m;
      g.N = st.n_is_n ? sc.n : sc.m;
      g.K = st.k_is_n ? sc.n : sc.m;
      g.count = sc.count;
      g.tiles_m = (g.M + tile_m - 1) / tile_m;
      g.tiles_n = (g.N + 255) / 256;
      g.tile_begin = tiles;
      canonical += 2.0 * g.count * double(g.M) * g.N * g.K;
      if (lean) {
        // every m x m buffer holds a symmetric iterate
        if (st.sym && st.out_buf >= MM0) g.lean |= kLeanOut;
        if (st.a_buf >= MM0) g.lean |= kLeanA;
        if (!st.b_mn && st.b_buf >= MM0) g.lean |= kLeanB;
      }
      if (st.sym) {
        g.sym = 1;
        g.tile_list = dtiles + tiles_off[tk][c];
        g.tiles_per_mat = static_cast<int32_t>(class_tiles[tk][c].size());
        tiles += int64_t(g.count) * g.tiles_per_mat;
        flops += g.count * tile_flops(class_tiles[tk][c], g.M, g.K, tile_m);
      } else {
        tiles += int64_t(g.count) * g.tiles_m * g.tiles_n;
        flops += 2.0 * g.count * double(g.M) * g.N * g.K;
      }
      gs[j] = g;
    }
    GemmLaunch l{};
    l.groups = reinterpret_cast<const GemmGroup*>(dbase + groups_off) + s * nclass;
    l.num_groups = nbig;
    l.b_mn_major = st.b_mn ? 1 : 0;
    l.has_aux = st.aux_buf >= 0 ? 1 : 0;
    l.fp16 = P.x_fp16 ? 1 : 0;
    l.pair = pair ? 1 : 0;
    for (int j = 0; j < nbig && pair; ++j) {
      const int r = gs[j].N % 256;
      if (r != 0 && r <= 128) l.narrow = 1;
    }
    l.total_tiles = tiles;
    l.alpha = st.alpha;
    l.beta = st.beta;
    l.diag = st.diag;
    l.flops = flops;
    l.canonical_flops = canonical;
    P.launches.push_back(l);
  }

  if (sink) {
    // pageable source: the copy is staged before cudaMemcpyAsync returns
    e = cudaMemcpyAsync(P.dmeta, host.data(), total, cudaMemcpyHostToDevice, sink->stream);
  } else {
    e = cudaMemcpy(P.dmeta, host.data(), total, cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) return fail_cuda(e, "copy plan metadata");
  (void)ws_bytes;
  return NSM_OK;
}

struct PlanCache {
  std::mutex mu;
  std::list<std::pair<std::string, std::unique_ptr<Plan>>> lru;  // front = most recent
  static constexpr size_t kMax = 8;
};

PlanCache& cache() {
  static PlanCache* c = new PlanCache();  // never destroyed: plans may outlive static teardown
  return *c;
}

std::string plan_key(int device, const int32_t* shapes, const int64_t* offsets, int n, int method,
                     int steps, const void* ws) {
  std::string k;
  k.reserve(64 + size_t(n) * 16);
  auto put = [&](const void* p, size_t b) { k.append(static_cast<const char*>(p), b); };
  const int opts = (pair_kernels_enabled() ? 1 : 0) | (small_kernel_enabled() ? 2 : 0) |
                   (lean_storage_enabled() ? 4 : 0);
  put(&device, sizeof(device));
  put(&opts, sizeof(opts));
  put(&method, sizeof(method));
  put(&steps, sizeof(steps));
  put(&n, sizeof(n));
  put(&ws, sizeof(ws));
  put(shapes, sizeof(int32_t) * 2 * size_t(n));
  put(offsets, sizeof(int64_t) * size_t(n));
  return k;
}

// Returns a plan (owned by the cache) or NULL with the error set.
Plan* get_plan(const int32_t* shapes, const int64_t* offsets, int n, int method, int steps, void* ws,
               size_t ws_bytes, int* rc) {
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) {
    *rc = fail_cuda(e, "cudaGetDevice");
    return nullptr;
  }
  const std::string key = plan_key(device, shapes, offsets, n, method, steps, ws);
  PlanCache& C = cache();
  std::lock_guard<std::mutex> lock(C.mu);
  for (auto it = C.lru.begin(); it != C.lru.end(); ++it) {
    if (it->first == key) {
      C.lru.splice(C.lru.begin(), C.lru, it);
      return C.lru.front().second.get();
    }
  }
  std::unique_ptr<Plan> P(new Plan());
  P->device = device;
  *rc = build_plan(*P, shapes, offsets, n, method, steps, ws, ws_bytes);
  if (*rc != NSM_OK) return nullptr;
  if (C.lru.size() >= PlanCache::kMax) {
    // the evicted plan's metadata may still be read by queued kernels
    cudaDeviceSynchronize();
    C.lru.pop_back();
  }
  C.lru.emplace_front(key, std::move(P));
  return C.lru.front().second.get();
}

// ---------------------------------------------------------------- timing

// Kernel kinds the timing hooks distinguish (NSM_KIND_* in the header).
constexpr int kKinds = 8;

struct Timing {
  std::mutex mu;
  bool enabled = false;
  struct Rec {
    cudaEvent_t a, b;
    int kind;
    double work;
  };
  std::vector<Rec> pending;
  std::vector<cudaEvent_t> pool;
  double ms[kKinds] = {0}, work[kKinds] = {0};
  int64_t launches[kKinds] = {0};
  cudaEvent_t get() {
    if (!pool.empty()) {
      cudaEvent_t e = pool.back();
      pool.pop_back();
      return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
  }
  void collect() {
    for (auto& r : pending) {
      cudaEventSynchronize(r.b);
      float t = 0.f;
      cudaEventElapsedTime(&t, r.a, r.b);
      ms[r.kind] += t;
      work[r.kind] += r.work;
      launches[r.kind] += 1;
      pool.push_back(r.a);
      pool.push_back(r.b);
    }
    pending.clear();
  }
};

Timing& timing() {
  static Timing* t = new Timing();
  return *t;
}

// Brackets one launch with events on `stream` while timing is enabled.
class TimedLaunch {
 public:
  TimedLaunch(cudaStream_t stream, int kind, double work) : stream_(stream), kind_(kind), work_(work) {
    Timing& T = timing();
    std::lock_guard<std::mutex> lock(T.mu);
    if (!T.enabled) return;
    a_ = T.get();
    b_ = T.get();
    cudaEventRecord(a_, stream_);
  }
  ~TimedLaunch() {
    if (!a_) return;
    Timing& T = timing();
    std::lock_guard<std::mutex> lock(T.mu);
    cudaEventRecord(b_, stream_);
    T.pending.push_back({a_, b_, kind_, work_});
  }

 private:
  cudaStream_t stream_;
  int kind_;
  double work_;
  cudaEvent_t a_ = nullptr, b_ = nullptr;
};

// ---------------------------------------------------------------- validation helpers

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int validate_offsets(const int64_t* offsets, const int32_t* shapes, int n, int64_t* extent) {
  if (!offsets) return fail(NSM_ERR_NULL, "offsets is NULL");
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) {
    if (offsets[i] < 0) return fail(NSM_ERR_OFFSET, "offset %d is negative", i);
    if (offsets[i] % 8 != 0) return fail(NSM_ERR_ALIGN, "offset %d (%lld) is not a multiple of 8 elements", i, (long long)offsets[i]);
    order[i] = i;
  }
  std::sort(order.begin(), order.end(), [&](int a, int b) { return offsets[a] < offsets[b]; });
  int64_t end_prev = 0;
  int64_t ext = 0;
  for (int k = 0; k < n; ++k) {
    const int i = order[k];
    const int64_t len = int64_t(shapes[2 * i]) * shapes[2 * i + 1];
    if (k > 0 && offsets[i] < end_prev) return fail(NSM_ERR_OFFSET, "matrix %d overlaps the matrix before it", i);
    end_prev = offsets[i] + len;
    ext = std::max(ext, end_prev);
  }
  *extent = ext;
  return NSM_OK;
}

bool ranges_overlap(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + bn && b0 < a0 + an;
}

// The address the kernels use for a buffer: device (or managed) memory as it is,
// page-locked host memory through its device mapping (read or written in place over the
// host link).  Pageable host memory is refused here instead of faulting a kernel.
int device_view(const void* p, const char* what, const void** out) {
  cudaPointerAttributes a{};
  const cudaError_t e = cudaPointerGetAttributes(&a, p);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail(NSM_ERR_ARG, "%s: cudaPointerGetAttributes failed (%s)", what, cudaGetErrorString(e));
  }
  if (a.type == cudaMemoryTypeUnregistered)
    return fail(NSM_ERR_ARG, "%s is neither device memory nor page-locked host memory", what);
  if (a.type == cudaMemoryTypeHost) {
    if (!a.devicePointer) return fail(NSM_ERR_ARG, "%s is page-locked host memory without a device mapping", what);
    *out = a.devicePointer;
  } else {
    *out = p;
  }
  return NSM_OK;
}

// The orthogonalisation's input and output, as device_view gives them, 16-byte aligned.
int device_views(const void* in_bf16, const void* out_bf16, const void** in, const void** out) {
  int rc = device_view(in_bf16, "in_bf16", in);
  if (rc != NSM_OK) return rc;
  rc = device_view(out_bf16, "out_bf16", out);
  if (rc != NSM_OK) return rc;
  if (!aligned(*in, 16) || !aligned(*out, 16)) return fail(NSM_ERR_ALIGN, "a device mapping is not 16-byte aligned");
  return NSM_OK;
}

int check_workspace(void* ws, size_t ws_bytes, size_t need) {
  if (!ws) return fail(NSM_ERR_WORKSPACE, "workspace is NULL");
  if (!aligned(ws, 256)) return fail(NSM_ERR_ALIGN, "workspace is not 256-byte aligned");
  if (ws_bytes < need) return fail(NSM_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", ws_bytes, need);
  return NSM_OK;
}

// Launches the chain: the small-matrix kernel, then the grouped GEMMs.  Both leave O in
// the X buffer P.final_buf.
int run_chain(Plan& P, cudaStream_t stream, int* launches) {
  int num_sms = 0;
  cudaError_t e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, P.device);
  if (e != cudaSuccess) return fail_cuda(e, "cudaDeviceGetAttribute");
  if (P.n_small_jobs > 0) {
    TimedLaunch t(stream, NSM_KIND_SMALL, P.small_bytes);
    e = launch_ns_small(P.d_small_jobs, P.n_small_jobs, P.d_small_ops, P.n_small_ops, P.x_fp16 ? 1 : 0, num_sms,
                        stream);
    if (e != cudaSuccess) return fail_cuda(e, "small-matrix Newton-Schulz launch");
    ++*launches;
  }
  for (size_t k = 0; k < P.launches.size(); ++k) {
    const GemmLaunch& l = P.launches[k];
    TimedLaunch t(stream, NSM_KIND_GEMM, l.flops);
    e = launch_gemm(l, num_sms, stream);
    if (e != cudaSuccess) return fail_cuda(e, "Newton-Schulz GEMM launch");
    ++*launches;
  }
  return NSM_OK;
}

// The orthogonalisation of a plan's table: the sums and maxima of G per chunk, each
// matrix's s and exponent k, U = G stored as G 2^k, the chain, and the export of O.
int run_orthogonalize(Plan& P, const void* in_bf16, void* out_bf16, int n, cudaStream_t stream, int* launches) {
  char* ws = P.ws;
  const Layout& L = P.L;
  float* partials = reinterpret_cast<float*>(ws + L.off_partials);
  float* scales = reinterpret_cast<float*>(ws + L.off_scales);
  float* xs = reinterpret_cast<float*>(ws + L.off_xs);
  float* xs_cls = reinterpret_cast<float*>(ws + L.off_xs_cls);
  const double elems = double(P.elems);
  cudaError_t e;
  {
    TimedLaunch t(stream, NSM_KIND_GRAD_NORM, 2.0 * elems);
    e = launch_grad_norm(in_bf16, P.d_mats, n, L.total_chunks, partials, stream);
  }
  if (e != cudaSuccess) return fail_cuda(e, "norm launch");
  ++*launches;
  {
    TimedLaunch t(stream, NSM_KIND_NORM, 8.0 * double(L.total_chunks) + 12.0 * n);
    e = launch_scale_finalize(P.d_mats, n, partials, L.total_chunks, 0, nullptr, scales, nullptr, xs, xs_cls,
                              kNormEps, stream);
  }
  if (e != cudaSuccess) return fail_cuda(e, "norm launch");
  ++*launches;
  {
    TimedLaunch t(stream, NSM_KIND_LAYOUT, 4.0 * elems);
    e = launch_to_class(in_bf16, nullptr, 0, 0, 0.f, ws + L.off_x[0], P.x_fp16 ? 1 : 0, P.d_mats, n, L.total_tiles,
                        scales, nullptr, stream);
  }
  if (e != cudaSuccess) return fail_cuda(e, "layout launch");
  ++*launches;
  const int rc = run_chain(P, stream, launches);
  if (rc != NSM_OK) return rc;
  {
    TimedLaunch t(stream, NSM_KIND_APPLY, 4.0 * elems);
    e = launch_export(ws + L.off_x[P.final_buf], P.final_fp16 ? 1 : 0, P.final_is_input ? xs : nullptr, out_bf16,
                      P.d_mats, n, L.total_tiles, stream);
  }
  if (e != cudaSuccess) return fail_cuda(e, "export launch");
  ++*launches;
  return NSM_OK;
}

// ---------------------------------------------------------------- allocation-free path

// Device memory of the allocation-free orthogonalisation: its workspace and its launch
// plan.  It is part of the library's module, so every GPU that loads the library holds
// it until the process exits; no call ever allocates it.
constexpr size_t kNoAllocBytes = size_t(64) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocBytes];

// What the allocation-free path keeps per device: the context it belongs to, the array's
// device address in that context, and the plan whose metadata the array holds now (with
// the key it was built for), so that a call on the same table uploads nothing.
struct NoAllocState {
  unsigned long long ctx_id = 0;
  char* scratch = nullptr;
  std::string key;
  std::unique_ptr<Plan> plan;
};

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

// Unique id of the context current on this thread for `device` (a context created after
// a device reset gets a new id, so nothing looked up in the old one is used again).
int current_context_id(int device, unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  if (!get_current || !get_id) return fail(NSM_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId are unavailable");
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return fail(NSM_ERR_CUDA, "cuCtxGetCurrent failed");
  if (!ctx) {
    // this thread has not used the device yet: make its primary context current
    const cudaError_t e = cudaSetDevice(device);
    if (e != cudaSuccess) return fail_cuda(e, "cudaSetDevice");
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return fail(NSM_ERR_CUDA, "no current CUDA context");
  }
  if (get_id(ctx, id) != CUDA_SUCCESS) return fail(NSM_ERR_CUDA, "cuCtxGetId failed");
  return NSM_OK;
}

// The state of the current device, with the array's device address looked up (once per
// device and context, with that device current).  Called with noalloc_mutex() held.
NoAllocState* noalloc_state(int device, int* rc) {
  static NoAllocState states[64];
  if (device < 0 || device >= 64) {
    *rc = fail(NSM_ERR_CUDA, "device ordinal %d out of range", device);
    return nullptr;
  }
  unsigned long long id = 0;
  *rc = current_context_id(device, &id);
  if (*rc != NSM_OK) return nullptr;
  NoAllocState& st = states[device];
  if (!st.scratch || st.ctx_id != id) {
    st.plan.reset();
    st.key.clear();
    st.scratch = nullptr;
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) {
      *rc = fail_cuda(e, "cudaGetSymbolAddress(allocation-free scratch)");
      return nullptr;
    }
    st.scratch = static_cast<char*>(p);
    st.ctx_id = id;
  }
  return &st;
}

std::mutex& noalloc_mutex() {
  static std::mutex* mu = new std::mutex();
  return *mu;
}

}  // namespace

bool pdl_for_launches() { return t_pdl; }

int option_value(int option) {
  switch (option) {
    case NSM_OPT_PAIR_KERNELS: return g_opt_pair.load();
    case NSM_OPT_SMALL_KERNEL: return g_opt_small.load();
    case NSM_OPT_PDL: return g_opt_pdl.load();
    case NSM_OPT_SYM_STORAGE: return g_opt_lean.load();
    case NSM_OPT_BOUNDS_CHECKS: return kChecked ? 1 : 0;
    default: return -1;
  }
}

}  // namespace nsm

using namespace nsm;

extern "C" {

int nsm_version(void) { return 100; }

const char* nsm_last_error(void) { return t_last_error.c_str(); }

int nsm_last_launch_count(void) { return t_last_launches; }

int nsm_route(const char* name, int ndim) {
  if (!name) return fail(NSM_ERR_NULL, "name is NULL");
  if (ndim < 2) return 0;
  std::string s(name);
  for (char& ch : s) {
    if (ch >= 'A' && ch <= 'Z') ch = static_cast<char>(ch - 'A' + 'a');
  }
  if (s.find("embed") != std::string::npos) return 0;
  if (s.find("lm_head") != std::string::npos) return 0;
  return 1;
}

int nsm_input_exponent(float max_abs, int has_hint, int hint, int* k_out, int* next_out, int* store_out) {
  if (!k_out || !next_out || !store_out) return fail(NSM_ERR_NULL, "an output pointer is NULL");
  const InExponent r = in_exponent(max_abs, has_hint != 0, hint);
  *k_out = r.k;
  *next_out = r.next;
  *store_out = r.store;
  return NSM_OK;
}

int nsm_pack(const int32_t* shapes, int n, int64_t align_elems, int64_t* offsets_out, int64_t* total_out) {
  if (!offsets_out || !total_out) return fail(NSM_ERR_NULL, "output pointer is NULL");
  int rc = validate_shapes(shapes, n);
  if (rc != NSM_OK) return rc;
  if (align_elems < 1) return fail(NSM_ERR_ARG, "align_elems must be >= 1");
  int64_t cursor = 0;
  for (int i = 0; i < n; ++i) {
    offsets_out[i] = cursor;
    const int64_t end = cursor + int64_t(shapes[2 * i]) * shapes[2 * i + 1];
    cursor = (end + align_elems - 1) / align_elems * align_elems;
  }
  *total_out = cursor;
  return NSM_OK;
}

int nsm_assign_owners(const int32_t* shapes, int n, int world, int ns_method, int ns_steps, int32_t* owner_out,
                      int64_t* load_out) {
  if (!owner_out) return fail(NSM_ERR_NULL, "owner_out is NULL");
  int rc = validate_shapes(shapes, n);
  if (rc != NSM_OK) return rc;
  rc = validate_method(ns_method, ns_steps);
  if (rc != NSM_OK) return rc;
  if (world < 1 || world > (1 << 20)) return fail(NSM_ERR_ARG, "world = %d out of range", world);
  // cost of a matrix: flops of its Newton-Schulz chain (the step's dominant work)
  std::vector<int64_t> cost(n);
  for (int i = 0; i < n; ++i) {
    const int64_t r = shapes[2 * i], c = shapes[2 * i + 1];
    cost[i] = chain_flops(ns_method, ns_steps, std::min(r, c), std::max(r, c));
  }
  // longest processing time first: heaviest matrix to the least-loaded owner; ties go to
  // the lower matrix index and the lower rank, so every rank computes the same plan
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });
  std::vector<int64_t> load(world, 0);
  for (int i : order) {
    int best = 0;
    for (int w = 1; w < world; ++w) {
      if (load[w] < load[best]) best = w;
    }
    owner_out[i] = best;
    load[best] += cost[i];
  }
  if (load_out) std::copy(load.begin(), load.end(), load_out);
  return NSM_OK;
}

int nsm_workspace_iterate(const int32_t* shapes, int n, int ns_method, int ns_steps, int i, int buf,
                          size_t* offset_bytes, int* m_out, int* ld_out) {
  if (!offset_bytes || !m_out || !ld_out) return fail(NSM_ERR_NULL, "output pointer is NULL");
  int rc = validate_shapes(shapes, n);
  if (rc != NSM_OK) return rc;
  rc = validate_method(ns_method, ns_steps);
  if (rc != NSM_OK) return rc;
  if (i < 0 || i >= n) return fail(NSM_ERR_ARG, "matrix %d not in [0, %d)", i, n);
  const Layout L = make_layout(shapes, n, ns_method, ns_steps);
  if (buf < 0 || buf >= L.num_mm) return fail(NSM_ERR_ARG, "buffer %d not in [0, %d)", buf, L.num_mm);
  const ShapeClass& sc = L.classes[L.cls_of[i]];
  const bool small = ns_steps > 0 && small_kernel_enabled() && sc.m <= kSmallMaxM;
  *m_out = small ? 0 : sc.m;
  *ld_out = sc.ldm;
  *offset_bytes = L.off_mm[buf] + (size_t(sc.mm_base) + size_t(L.batch_of[i]) * sc.m * sc.ldm) * 2;
  return NSM_OK;
}

size_t muon_workspace_bytes(const int32_t* shapes, int n, int ns_method, int ns_steps) {
  if (validate_shapes(shapes, n) != NSM_OK) return 0;
  if (validate_method(ns_method, ns_steps) != NSM_OK) return 0;
  return make_layout(shapes, n, ns_method, ns_steps).bytes;
}

int muon_step(const void* packed_grads, float* packed_params, float* momentum, const int64_t* offsets,
              const int32_t* shapes, int n, float lr, float wd, float mu, int ns_method, int ns_steps,
              int nesterov, void* workspace, size_t workspace_bytes, nsm_stream_t stream_) {
  return muon_step_with_copy(packed_grads, packed_params, momentum, nullptr, offsets, shapes, n, lr, wd, mu,
                             ns_method, ns_steps, nesterov, workspace, workspace_bytes, stream_);
}

int muon_step_with_copy(const void* packed_grads, float* packed_params, float* momentum, void* params_bf16,
                        const int64_t* offsets, const int32_t* shapes, int n, float lr, float wd, float mu,
                        int ns_method, int ns_steps, int nesterov, void* workspace, size_t workspace_bytes,
                        nsm_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!packed_grads || !packed_params || !momentum) return fail(NSM_ERR_NULL, "a device buffer is NULL");
  int rc = validate_shapes(shapes, n);
  if (rc != NSM_OK) return rc;
  rc = validate_method(ns_method, ns_steps);
  if (rc != NSM_OK) return rc;
  if (!std::isfinite(lr) || !std::isfinite(wd) || !std::isfinite(mu))
    return fail(NSM_ERR_ARG, "lr, wd and mu must be finite");
  int64_t extent = 0;
  rc = validate_offsets(offsets, shapes, n, &extent);
  if (rc != NSM_OK) return rc;
  if (!aligned(packed_grads, 16) || !aligned(packed_params, 16) || !aligned(momentum, 16))
    return fail(NSM_ERR_ALIGN, "device buffers must be 16-byte aligned");
  if (ranges_overlap(packed_grads, size_t(extent) * 2, packed_params, size_t(extent) * 4) ||
      ranges_overlap(packed_grads, size_t(extent) * 2, momentum, size_t(extent) * 4) ||
      ranges_overlap(packed_params, size_t(extent) * 4, momentum, size_t(extent) * 4))
    return fail(NSM_ERR_ARG, "grads, params and momentum must not overlap");
  if (params_bf16) {
    if (!aligned(params_bf16, 16)) return fail(NSM_ERR_ALIGN, "the bf16 copy must be 16-byte aligned");
    if (ranges_overlap(params_bf16, size_t(extent) * 2, packed_grads, size_t(extent) * 2) ||
        ranges_overlap(params_bf16, size_t(extent) * 2, packed_params, size_t(extent) * 4) ||
        ranges_overlap(params_bf16, size_t(extent) * 2, momentum, size_t(extent) * 4))
      return fail(NSM_ERR_ARG, "the bf16 copy must not overlap grads, params or momentum");
  }
  const Layout L = make_layout(shapes, n, ns_method, ns_steps);
  rc = check_workspace(workspace, workspace_bytes, L.bytes);
  if (rc != NSM_OK) return rc;
  const void* grads = nullptr;  // the address the kernels read G at
  rc = device_view(packed_grads, "packed_grads", &grads);
  if (rc != NSM_OK) return rc;
  if (!aligned(grads, 16)) return fail(NSM_ERR_ALIGN, "packed_grads' device mapping is not 16-byte aligned");

  Plan* P = get_plan(shapes, offsets, n, ns_method, ns_steps, workspace, workspace_bytes, &rc);
  if (!P) return rc;
  const PdlScope pdl(P->elems);
  char* ws = P->ws;  // L (above) is the plan's layout
  float* tparts = reinterpret_cast<float*>(ws + L.off_tparts);
  float* scales = reinterpret_cast<float*>(ws + L.off_scales);
  float* xs = reinterpret_cast<float*>(ws + L.off_xs);
  float* xs_cls = reinterpret_cast<float*>(ws + L.off_xs_cls);
  int* hints = reinterpret_cast<int*>(ws + L.off_hints);
  int* redo = reinterpret_cast<int*>(ws + L.off_redo);
  int launches = 0;
  const double elems = double(P->elems);
  cudaError_t e;
  // One pass over G and M: M updated, U stored as U 2^k with each matrix's exponent hint
  // (the one the previous step on this table chose), per-tile sums and maxima of U.
  {
    TimedLaunch t(stream, NSM_KIND_MOMENTUM, 12.0 * elems);
    e = launch_momentum_class(grads, momentum, nesterov, mu, ws + L.off_x[0], P->x_fp16 ? 1 : 0, P->d_mats, n,
                              L.total_tiles, hints, tparts, redo, stream);
  }
  if (e != cudaSuccess) return fail_cuda(e, "momentum/layout launch");
  ++launches;
  // s and the exponent of each matrix; a hint that put max|U| 2^k outside the accepted
  // range marks its matrix for the layout pass below
  {
    TimedLaunch t(stream, NSM_KIND_NORM, 8.0 * kTileParts * double(L.total_tiles) + 16.0 * n);
    e = launch_scale_finalize(P->d_mats, n, tparts, L.total_tiles, 1, hints, scales, redo, xs, xs_cls, kNormEps,
                              stream);
  }
  if (e != cudaSuccess) return fail_cuda(e, "norm launch");
  ++launches;
  // U stored again where its hint was out of range (the first step on a table, or a jump
  // of the gradients' magnitude); every other matrix is skipped
  {
    TimedLaunch t(stream, NSM_KIND_LAYOUT, 0.0);
    e = launch_to_class(grads, momentum, 1, nesterov, mu, ws + L.off_x[0], P->x_fp16 ? 1 : 0, P->d_mats, n,
                        L.total_tiles, scales, redo, stream);
  }
  if (e != cudaSuccess) return fail_cuda(e, "layout launch");
  ++launches;
  // The chain leaves O in the workspace; the apply pass updates every matrix from it.
  rc = run_chain(*P, stream, &launches);
  if (rc != NSM_OK) return rc;
  {
    TimedLaunch t(stream, NSM_KIND_APPLY, (params_bf16 ? 12.0 : 10.0) * elems);
    e = launch_apply(ws + L.off_x[P->final_buf], P->final_fp16 ? 1 : 0, P->final_is_input ? xs : nullptr,
                     packed_params, params_bf16, P->d_mats, n, L.total_tiles, lr, wd, stream);
  }
  if (e != cudaSuccess) return fail_cuda(e, "apply launch");
  ++launches;
  t_last_launches = launches;
  return NSM_OK;
}

int muon_orthogonalize(const void* in_bf16, void* out_bf16, const int64_t* offsets, const int32_t* shapes, int n,
                       int ns_method, int ns_steps, void* workspace, size_t workspace_bytes, nsm_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!in_bf16 || !out_bf16) return fail(NSM_ERR_NULL, "a device buffer is NULL");
  int rc = validate_shapes(shapes, n);
  if (rc != NSM_OK) return rc;
  rc = validate_method(ns_method, ns_steps);
  if (rc != NSM_OK) return rc;
  int64_t extent = 0;
  rc = validate_offsets(offsets, shapes, n, &extent);
  if (rc != NSM_OK) return rc;
  if (!aligned(in_bf16, 16) || !aligned(out_bf16, 16)) return fail(NSM_ERR_ALIGN, "device buffers must be 16-byte aligned");
  if (ranges_overlap(in_bf16, size_t(extent) * 2, out_bf16, size_t(extent) * 2))
    return fail(NSM_ERR_ARG, "input and output must not overlap");
  const Layout L = make_layout(shapes, n, ns_method, ns_steps);
  rc = check_workspace(workspace, workspace_bytes, L.bytes);
  if (rc != NSM_OK) return rc;
  const void* in = nullptr;
  const void* out = nullptr;
  rc = device_views(in_bf16, out_bf16, &in, &out);
  if (rc != NSM_OK) return rc;

  Plan* P = get_plan(shapes, offsets, n, ns_method, ns_steps, workspace, workspace_bytes, &rc);
  if (!P) return rc;
  const PdlScope pdl(P->elems);
  int launches = 0;
  rc = run_orthogonalize(*P, in, const_cast<void*>(out), n, stream, &launches);
  if (rc != NSM_OK) return rc;
  t_last_launches = launches;
  return NSM_OK;
}

int adamw_step(const void* grads, float* params, float* exp_avg, float* exp_avg_sq, int64_t numel, float lr,
               float beta1, float beta2, float eps, float wd, int step, nsm_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (numel < 0) return fail(NSM_ERR_SHAPE, "numel is negative");
  if (numel == 0) {
    t_last_launches = 0;
    return NSM_OK;
  }
  if (!grads || !params || !exp_avg || !exp_avg_sq) return fail(NSM_ERR_NULL, "a device buffer is NULL");
  if (step < 1) return fail(NSM_ERR_ARG, "step counts from 1");
  if (!(beta1 >= 0.f && beta1 < 1.f) || !(beta2 >= 0.f && beta2 < 1.f))
    return fail(NSM_ERR_ARG, "betas must lie in [0, 1)");
  if (!std::isfinite(lr) || !std::isfinite(wd) || !(eps >= 0.f) || !std::isfinite(eps))
    return fail(NSM_ERR_ARG, "lr, wd, eps must be finite (eps >= 0)");
  if (!aligned(grads, 16) || !aligned(params, 16) || !aligned(exp_avg, 16) || !aligned(exp_avg_sq, 16))
    return fail(NSM_ERR_ALIGN, "device buffers must be 16-byte aligned");
  const size_t fb = size_t(numel) * 4;
  if (ranges_overlap(params, fb, exp_avg, fb) || ranges_overlap(params, fb, exp_avg_sq, fb) ||
      ranges_overlap(exp_avg, fb, exp_avg_sq, fb) || ranges_overlap(grads, size_t(numel) * 2, params, fb))
    return fail(NSM_ERR_ARG, "AdamW buffers must not overlap");
  const PdlScope pdl(numel);
  const double bc1 = 1.0 - std::pow(double(beta1), double(step));
  const double bc2 = 1.0 - std::pow(double(beta2), double(step));
  cudaError_t e;
  {
    TimedLaunch t(stream, NSM_KIND_ADAMW, 26.0 * double(numel));
    e = launch_adamw(grads, params, exp_avg, exp_avg_sq, numel, lr, beta1, beta2, eps, wd, static_cast<float>(bc1),
                     static_cast<float>(bc2), stream);
  }
  if (e != cudaSuccess) return fail_cuda(e, "AdamW launch");
  t_last_launches = 1;
  return NSM_OK;
}

int nsm_gemm(const void* a, int lda, const void* b, int ldb, void* out, int ldo, const void* aux, int ldx, int M,
             int N, int K, int b_mn_major, int fp16, int flags, float alpha, float beta, float diag,
             void* scratch, size_t scratch_bytes, nsm_stream_t stream_) {
  const bool symmetric = (flags & NSM_GEMM_SYMMETRIC) != 0;
  const bool pair = (flags & NSM_GEMM_PAIR) != 0;
  const int tile_m = pair ? 256 : 128;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!a || !b || !out || !scratch) return fail(NSM_ERR_NULL, "a, b, out and scratch must be non-NULL");
  if (M <= 0 || N <= 0 || K <= 0 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return fail(NSM_ERR_SHAPE, "bad GEMM shape %dx%dx%d", M, N, K);
  const int b_cols = b_mn_major ? N : K;
  if (lda < K || ldb < b_cols || ldo < N || (aux && ldx < N))
    return fail(NSM_ERR_SHAPE, "a row stride is shorter than its row");
  if (lda % 8 || ldb % 8 || ldo % 8 || (aux && ldx % 8))
    return fail(NSM_ERR_ALIGN, "row strides must be multiples of 8 elements");
  if (!aligned(a, 16) || !aligned(b, 16) || !aligned(out, 16) || (aux && !aligned(aux, 16)))
    return fail(NSM_ERR_ALIGN, "pointers must be 16-byte aligned");
  if (!aligned(scratch, 128)) return fail(NSM_ERR_ALIGN, "scratch must be 128-byte aligned");
  if (symmetric && M != N) return fail(NSM_ERR_SHAPE, "a symmetric output needs M == N");
  const std::vector<int32_t> sym_tiles = symmetric ? upper_tiles(M, tile_m) : std::vector<int32_t>();
  const size_t need = nsm_gemm_scratch_bytes(M, N, flags);
  if (scratch_bytes < need) return fail(NSM_ERR_WORKSPACE, "scratch needs %zu bytes", need);
  if (aux && ranges_overlap(aux, size_t(M) * ldx * 2, out, size_t(M) * ldo * 2))
    return fail(NSM_ERR_ARG, "aux must not overlap out");
  struct Blob {
    CUtensorMap ma, mb, mo, mbn;
    GemmGroup g;
  };
  static_assert(sizeof(Blob) <= 1024, "scratch blob");
  Blob blob;
  std::memset(&blob, 0, sizeof(blob));
  const int a_box = 128;
  const int b_box = b_mn_major ? (pair ? 128 : 64) : (pair ? 128 : 256);
  int rc = encode_map(&blob.ma, const_cast<void*>(a), fp16 != 0, K, M, lda, 1, nullptr, nullptr, a_box);
  if (rc != NSM_OK) return rc;
  if (b_mn_major) rc = encode_map(&blob.mb, const_cast<void*>(b), fp16 != 0, N, K, ldb, 1, nullptr, nullptr, b_box);
  else rc = encode_map(&blob.mb, const_cast<void*>(b), fp16 != 0, K, N, ldb, 1, nullptr, nullptr, b_box);
  if (rc != NSM_OK) return rc;
  if (!b_mn_major) {
    rc = encode_map(&blob.mbn, const_cast<void*>(b), fp16 != 0, K, N, ldb, 1, nullptr, nullptr, 64);
    if (rc != NSM_OK) return rc;
  }
  // TMA stores write whole 16-byte units of a row: only for rows of a multiple of 8
  const bool tma_store = N % 8 == 0;
  if (tma_store) {
    rc = encode_map(&blob.mo, out, fp16 != 0, N, M, ldo, 1, nullptr, nullptr, 64, true);
    if (rc != NSM_OK) return rc;
  }
  Blob* d = static_cast<Blob*>(scratch);
  GemmGroup& g = blob.g;
  g.map_a = &d->ma;
  g.map_b = &d->mb;
  g.map_b_narrow = b_mn_major ? &d->mb : &d->mbn;
  g.map_out = tma_store ? &d->mo : nullptr;
  g.out = out;
  g.aux = aux;
  g.ld_out = ldo;
  g.ld_aux = aux ? ldx : 0;
  g.M = M;
  g.N = N;
  g.K = K;
  g.count = 1;
  g.tiles_m = (M + tile_m - 1) / tile_m;
  g.tiles_n = (N + 255) / 256;
  g.tile_begin = 0;
  g.a_box = a_box;
  g.b_box = b_box;
  std::vector<uint8_t> host(sizeof(Blob) + sym_tiles.size() * sizeof(int32_t));
  if (symmetric) {
    g.sym = 1;
    g.tiles_per_mat = static_cast<int32_t>(sym_tiles.size());
    g.tile_list = reinterpret_cast<const int32_t*>(static_cast<char*>(scratch) + sizeof(Blob));
    std::memcpy(host.data() + sizeof(Blob), sym_tiles.data(), sym_tiles.size() * sizeof(int32_t));
  }
  std::memcpy(host.data(), &blob, sizeof(Blob));
  cudaError_t e = cudaMemcpyAsync(scratch, host.data(), host.size(), cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return fail_cuda(e, "copy GEMM descriptors");
  // the source is pageable host memory: the copy is staged before cudaMemcpyAsync returns
  GemmLaunch l{};
  l.groups = &d->g;
  l.num_groups = 1;
  l.b_mn_major = b_mn_major ? 1 : 0;
  l.has_aux = aux ? 1 : 0;
  l.fp16 = fp16 ? 1 : 0;
  l.pair = pair ? 1 : 0;
  l.narrow = (pair && N % 256 != 0 && N % 256 <= 128) ? 1 : 0;
  l.total_tiles = symmetric ? int64_t(sym_tiles.size()) : int64_t(g.tiles_m) * g.tiles_n;
  l.alpha = alpha;
  l.beta = aux ? beta : 0.f;
  l.diag = diag;
  l.canonical_flops = 2.0 * M * double(N) * K;
  l.flops = symmetric ? tile_flops(sym_tiles, M, K, tile_m) : l.canonical_flops;
  int dev = 0, num_sms = 0;
  e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return fail_cuda(e, "device query");
  const PdlScope pdl(int64_t(M) * N);
  {
    TimedLaunch t(stream, NSM_KIND_GEMM, l.flops);
    e = launch_gemm(l, num_sms, stream);
  }
  if (e != cudaSuccess) return fail_cuda(e, "GEMM launch");
  t_last_launches = 1;
  return NSM_OK;
}

size_t nsm_gemm_scratch_bytes(int M, int N, int flags) {
  size_t b = 4 * sizeof(CUtensorMap) + sizeof(GemmGroup);
  if ((flags & NSM_GEMM_SYMMETRIC) && M > 0 && M == N)
    b += upper_tiles(M, (flags & NSM_GEMM_PAIR) ? 256 : 128).size() * sizeof(int32_t);
  return align_up(b, 128);
}

int muon_orthogonalize_noalloc(const void* in_bf16, void* out_bf16, const int64_t* offsets, const int32_t* shapes,
                               int n, int ns_method, int ns_steps, nsm_stream_t stream_) {
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (!in_bf16 || !out_bf16) return fail(NSM_ERR_NULL, "a device buffer is NULL");
  int rc = validate_shapes(shapes, n);
  if (rc != NSM_OK) return rc;
  rc = validate_method(ns_method, ns_steps);
  if (rc != NSM_OK) return rc;
  int64_t extent = 0;
  rc = validate_offsets(offsets, shapes, n, &extent);
  if (rc != NSM_OK) return rc;
  if (!aligned(in_bf16, 16) || !aligned(out_bf16, 16)) return fail(NSM_ERR_ALIGN, "device buffers must be 16-byte aligned");
  if (ranges_overlap(in_bf16, size_t(extent) * 2, out_bf16, size_t(extent) * 2))
    return fail(NSM_ERR_ARG, "input and output must not overlap");
  const size_t ws_bytes = make_layout(shapes, n, ns_method, ns_steps).bytes;
  if (ws_bytes >= kNoAllocBytes)
    return fail(NSM_ERR_WORKSPACE,
                "the allocation-free path holds %zu bytes; this table needs %zu bytes of workspace (use "
                "muon_orthogonalize with a caller workspace)",
                kNoAllocBytes, ws_bytes);
  const void* in = nullptr;
  const void* out = nullptr;
  rc = device_views(in_bf16, out_bf16, &in, &out);
  if (rc != NSM_OK) return rc;
  int device = 0;
  cudaError_t e = cudaGetDevice(&device);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  std::lock_guard<std::mutex> lock(noalloc_mutex());
  NoAllocState* st = noalloc_state(device, &rc);
  if (!st) return rc;
  char* scratch = st->scratch;

  // Workspace at the start of the array, the plan's metadata after it.  The kernels write
  // only the workspace, so the metadata of the last plan uploaded stays valid, and a call
  // on the same table (same key) reuses it without copying anything.
  const std::string key = plan_key(device, shapes, offsets, n, ns_method, ns_steps, scratch);
  if (!st->plan || st->key != key) {
    st->plan.reset();
    st->key.clear();
    std::unique_ptr<Plan> P(new Plan());
    P->device = device;
    const size_t meta_off = align_up(ws_bytes, kAlign);
    MetaSink sink{scratch + meta_off, kNoAllocBytes - meta_off, stream};
    rc = build_plan(*P, shapes, offsets, n, ns_method, ns_steps, scratch, ws_bytes, &sink);
    if (rc != NSM_OK) return rc;
    st->plan = std::move(P);
    st->key = key;
  }
  Plan& P = *st->plan;
  const PdlScope pdl(P.elems);
  int launches = 0;
  rc = run_orthogonalize(P, in, const_cast<void*>(out), n, stream, &launches);
  if (rc != NSM_OK) return rc;
  t_last_launches = launches;
  return NSM_OK;
}

int nsm_device_status(nsm_stream_t stream, int* status_out) {
  return nsm_device_status_detail(stream, status_out, nullptr, nullptr, nullptr);
}

int nsm_device_status_detail(nsm_stream_t stream_, int* status_out, int* kernel_out, int* role_out,
                             int* site_out) {
  if (!status_out) return fail(NSM_ERR_NULL, "status_out is NULL");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
  int* p = device_status_ptr();
  if (!p) return fail(NSM_ERR_CUDA, "device status word unavailable");
  int v = 0;
  e = cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fail_cuda(e, "read device status");
  const int zero = 0;
  e = cudaMemcpy(p, &zero, sizeof(int), cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return fail_cuda(e, "clear device status");
  const int kind = v & 0xff;
  const bool set = kind == kDevTimeout || kind == kDevBounds;
  *status_out = kind == kDevTimeout ? NSM_ERR_TIMEOUT : (kind == kDevBounds ? NSM_ERR_BOUNDS : NSM_OK);
  if (kernel_out) *kernel_out = set ? (v >> 8) & 0xff : 0;
  if (role_out) *role_out = set ? (v >> 16) & 0xff : 0;
  if (site_out) *site_out = set ? (v >> 24) & 0xff : 0;
  return NSM_OK;
}

int nsm_set_option(int option, int value) {
  if (option == NSM_OPT_BOUNDS_CHECKS) return fail(NSM_ERR_ARG, "NSM_OPT_BOUNDS_CHECKS is read only");
  const int max_value = option == NSM_OPT_PDL ? 2 : 1;
  if (value < 0 || value > max_value) return fail(NSM_ERR_ARG, "option value %d is not in [0, %d]", value, max_value);
  switch (option) {
    case NSM_OPT_PAIR_KERNELS: g_opt_pair.store(value); return NSM_OK;
    case NSM_OPT_SMALL_KERNEL: g_opt_small.store(value); return NSM_OK;
    case NSM_OPT_PDL: g_opt_pdl.store(value); return NSM_OK;
    case NSM_OPT_SYM_STORAGE: g_opt_lean.store(value); return NSM_OK;
    default: return fail(NSM_ERR_ARG, "unknown option %d", option);
  }
}

int nsm_get_option(int option) {
  const int v = nsm::option_value(option);
  return v >= 0 ? v : fail(NSM_ERR_ARG, "unknown option %d", option);
}

int nsm_status_selftest(int wait_us, nsm_stream_t stream_) {
  if (wait_us < 1 || wait_us > 2000000) return fail(NSM_ERR_ARG, "wait_us = %d not in [1, 2000000]", wait_us);
  const cudaError_t e = launch_status_selftest(uint64_t(wait_us) * 1000u, reinterpret_cast<cudaStream_t>(stream_));
  if (e != cudaSuccess) return fail_cuda(e, "status self-test launch");
  return NSM_OK;
}

int nsm_copy_to_device(void* dst, const void* src, size_t bytes, int ctas, nsm_stream_t stream_) {
  if (!dst || !src) return fail(NSM_ERR_NULL, "dst or src is NULL");
  if (!aligned(dst, 16) || !aligned(src, 16)) return fail(NSM_ERR_ALIGN, "dst and src must be 16-byte aligned");
  if (ctas < 0 || ctas > 1024) return fail(NSM_ERR_ARG, "ctas = %d not in [0, 1024]", ctas);
  if (bytes == 0) return NSM_OK;
  // only page-locked host memory with a device mapping: anything else is refused before
  // a launch
  cudaPointerAttributes attr{};
  cudaError_t e = cudaPointerGetAttributes(&attr, src);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return fail_cuda(e, "cudaPointerGetAttributes(src)");
  }
  if (attr.type != cudaMemoryTypeHost || attr.devicePointer == nullptr)
    return fail(NSM_ERR_ARG, "src is not page-locked host memory with a device mapping");
  if (!aligned(attr.devicePointer, 16)) return fail(NSM_ERR_ALIGN, "src's device mapping is not 16-byte aligned");
  e = launch_copy_h2d(dst, attr.devicePointer, bytes, ctas ? ctas : 16, reinterpret_cast<cudaStream_t>(stream_));
  if (e != cudaSuccess) return fail_cuda(e, "copy launch");
  return NSM_OK;
}

int nsm_bounds_selftest(nsm_stream_t stream_) {
  const cudaError_t e = launch_bounds_selftest(reinterpret_cast<cudaStream_t>(stream_));
  if (e != cudaSuccess) return fail_cuda(e, "bounds self-test launch");
  return NSM_OK;
}

int nsm_timing_enable(int enable) {
  Timing& T = timing();
  std::lock_guard<std::mutex> lock(T.mu);
  T.enabled = enable != 0;
  return NSM_OK;
}

int nsm_timing_read(double* gemm_ms, int64_t* gemm_launches, double* gemm_flops) {
  return nsm_timing_read_kind(NSM_KIND_GEMM, gemm_ms, gemm_launches, gemm_flops);
}

int nsm_timing_read_kind(int kind, double* ms, int64_t* launches, double* work) {
  if (kind < 0 || kind >= kKinds) return fail(NSM_ERR_ARG, "unknown timing kind %d", kind);
  Timing& T = timing();
  std::lock_guard<std::mutex> lock(T.mu);
  T.collect();
  if (ms) *ms = T.ms[kind];
  if (launches) *launches = T.launches[kind];
  if (work) *work = T.work[kind];
  return NSM_OK;
}

int nsm_timing_reset(void) {
  Timing& T = timing();
  std::lock_guard<std::mutex> lock(T.mu);
  T.collect();
  for (int k = 0; k < kKinds; ++k) {
    T.ms[k] = 0;
    T.work[k] = 0;
    T.launches[k] = 0;
  }
  return NSM_OK;
}

}  // extern "C"
