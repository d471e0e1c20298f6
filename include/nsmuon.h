/*
 * nsmuon.h — C ABI of the GB300 (sm_103a) owner-side Muon optimizer step.
 *
 * One shared library, libnsmuon.so.  Every entry point takes plain pointers and sizes;
 * no framework types cross this boundary.  All device work is launched asynchronously
 * on the stream the caller passes (NULL = the legacy default stream).
 *
 * Sources (web pages, cited by title and section):
 *   [DSM]  "DeepSpeed 集成 Muon 优化器实战：从正交化原理到 ZeRO 微调配置"
 *   [DMZ]  "Z2 与 Z3 模式" (DMuon guide)
 *
 * Conventions shared by every call
 *   - Return value: NSM_OK (0) on success, a negative NSM_ERR_* code otherwise.  When
 *     argument validation fails nothing is launched and nsm_last_error() describes why.
 *     Kernel launches are asynchronous: a fault inside a kernel surfaces at the next
 *     synchronising CUDA call, and a bounded wait that expired inside a kernel is
 *     reported by nsm_device_status().
 *   - Ownership: the caller owns every buffer (device memory, host tables, workspace,
 *     stream).  Host tables are read during the call only.  The library keeps a small
 *     cache of launch plans (tensor maps and work lists, in device memory it allocates
 *     itself on the first call for a given table/workspace pair); it never frees or
 *     writes anything the caller owns except the documented outputs and the workspace.
 *     Because building a plan allocates, the first call for a new table/workspace pair
 *     should not be made inside CUDA stream capture.
 *   - Packed layout: a Muon group is one contiguous buffer; matrix i (rows x cols,
 *     row-major) starts at element offsets[i].  Offsets must be multiples of 8 elements,
 *     matrices must not overlap, and every base pointer must be 16-byte aligned.
 *   - shapes is a host array of n pairs {rows, cols} (int32, rows-then-cols).
 *   - Not thread-safe per workspace: two calls that share a workspace must be ordered
 *     on one stream.
 */
#ifndef NSMUON_H
#define NSMUON_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI-compatible with cudaStream_t / CUstream. */
typedef struct CUstream_st* nsm_stream_t;

#define NSM_OK             0
#define NSM_ERR_NULL      -1  /* a required pointer is NULL */
#define NSM_ERR_SHAPE     -2  /* n <= 0, rows or cols <= 0, or a size overflows */
#define NSM_ERR_OFFSET    -3  /* offsets overlap, are negative or not increasing */
#define NSM_ERR_ALIGN     -4  /* pointer or offset misaligned */
#define NSM_ERR_METHOD    -5  /* unknown ns_method or ns_steps out of [0, 16] */
#define NSM_ERR_WORKSPACE -6  /* workspace NULL or smaller than muon_workspace_bytes() */
#define NSM_ERR_CUDA      -7  /* a CUDA runtime/driver call failed */
#define NSM_ERR_TIMEOUT   -8  /* a bounded in-kernel wait expired (nsm_device_status) */
#define NSM_ERR_ARG       -9  /* any other invalid argument */
#define NSM_ERR_BOUNDS   -10  /* (checked build) a kernel's bounds check failed and the
                                 access was skipped (nsm_device_status) */

/* Newton-Schulz methods [DSM §核心算子].  Every form accumulates in fp32 on the tensor
 * cores; they differ in the half precision the iterates are stored in. */
#define NSM_NS_STANDARD      0  /* quintic steps on X, fp16 storage */
#define NSM_NS_GRAM          1  /* gram form on R = X X^T, fp16, re-anchored every 3 steps */
#define NSM_NS_STANDARD_BF16 2  /* quintic steps on X, bf16 storage (the page's stable form) */

/* Library version as MAJOR*10000 + MINOR*100 + PATCH. */
int nsm_version(void);

/* Message of the last failing call on this host thread ("" if none).  The pointer
 * stays valid until the next library call on the same thread. */
const char* nsm_last_error(void);

/* Routing rule of [DSM] §use_muon参数打标: returns 1 (Muon group) when ndim >= 2 and the
 * lower-cased name contains neither "embed" nor "lm_head", 0 (AdamW group) otherwise,
 * NSM_ERR_NULL if name is NULL.  name: NUL-terminated, ASCII case folding only.
 * Host-only; touches no GPU. */
int nsm_route(const char* name, int ndim);

/* Packed-buffer layout of [DMZ] §两种packed buffer生命周期 (one contiguous buffer per
 * owner): offsets_out[i] = start of matrix i, each rounded up to a multiple of
 * align_elems (>= 1, a multiple of 8 keeps the buffers usable by muon_step);
 * *total_out = end of the last matrix rounded up likewise.  offsets_out has n entries
 * (caller-allocated).  Host-only. */
int nsm_pack(const int32_t* shapes, int n, int64_t align_elems,
             int64_t* offsets_out, int64_t* total_out);

/* The exponent rule of muon_step's stored input (host-only; the kernels apply the same
 * function).  A matrix's normalised input is held as U 2^k rounded once to the storage
 * format; max_abs is its largest |U|.  With has_hint != 0 (the step), U was stored with
 * 2^hint (hint clamped to [-120, 120]): *store_out = 0 and *k_out = hint when
 * max_abs 2^hint lies in [2^4, 2^15), else *store_out = 1 and *k_out the exponent that
 * puts max_abs 2^k in [2^11, 2^12).  With has_hint == 0 (the orthogonalisation) *k_out
 * is that exponent and *store_out = 1.  *next_out is the hint the step leaves for its
 * next call: that exponent, or the hint when max_abs is 0, infinite or NaN (no exponent
 * follows from it; *k_out is then the hint, or 0).  Returns NSM_ERR_NULL for a NULL
 * output. */
int nsm_input_exponent(float max_abs, int has_hint, int hint, int* k_out, int* next_out, int* store_out);

/* Dedicated ownership ([DMZ] §两种packed buffer生命周期 and §每步通信字节数: every
 * Muon-target matrix has one owner, which alone runs its Newton-Schulz chain).  Assigns
 * the n matrices of a table to `world` owners by longest-processing-time-first on the
 * flops of each matrix's chain (ns_method/ns_steps as in muon_step): heaviest first, to
 * the least-loaded owner, ties to the lower rank.  Deterministic: every rank computes
 * the same plan.  owner_out: n int32 (host, caller-allocated); load_out: world int64
 * flops per owner, or NULL.  Host-only. */
int nsm_assign_owners(const int32_t* shapes, int n, int world, int ns_method, int ns_steps,
                      int32_t* owner_out, int64_t* load_out);

/* Layout query (host-only; for checks and debugging): where muon_step and
 * muon_orthogonalize keep matrix i's m x m iterates in the workspace.  Every m x m iterate
 * of the chain (A and B of the standard forms; R, H, Q and T of the gram form) is
 * symmetric, and the library stores it exactly symmetric: whole, or (NSM_OPT_SYM_STORAGE,
 * where every grouped launch runs on the 2-SM kernel) as its 256 x 256 tiles on and above
 * the diagonal, the diagonal tiles exactly symmetric and the rest of the block never
 * written.  buf selects one of the m x m
 * buffers: 0..1 for NSM_NS_STANDARD and NSM_NS_STANDARD_BF16, 0..3 for NSM_NS_GRAM.  On
 * return, *offset_bytes is the byte offset of matrix i's block in that buffer, *m its
 * order (m = min(rows, cols)) and *ld its row stride in 16-bit elements (fp16, or bf16
 * for NSM_NS_STANDARD_BF16).  *m = 0 when matrix i's chain runs in the small-matrix
 * kernel, whose iterates never leave shared memory.  Returns NSM_ERR_ARG for i or buf out
 * of range. */
int nsm_workspace_iterate(const int32_t* shapes, int n, int ns_method, int ns_steps, int i,
                          int buf, size_t* offset_bytes, int* m, int* ld);

/* Bytes of device workspace muon_step / muon_orthogonalize need for this table and
 * method (independent of offsets).  Returns 0 when the arguments are invalid (the
 * reason is in nsm_last_error()).  Host-only. */
size_t muon_workspace_bytes(const int32_t* shapes, int n, int ns_method, int ns_steps);

/* One owner-side Muon step over a packed group ([DSM] §什么是 Muon 优化器？,
 * §核心算子; [DMZ] §两种packed buffer生命周期), for every matrix i:
 *     M <- mu*M + G;   U = G + mu*M (nesterov != 0) or U = M (nesterov == 0)
 *     X = U / (||U||_F + 1e-7), working on U^T when rows > cols
 *     X <- ns_steps quintic Newton-Schulz steps (a, b, c) = (3.4445, -4.7750, 2.0315)
 *          in the standard or gram form (ns_method: NSM_NS_*)
 *     p <- p*(1 - lr*wd) - lr*sqrt(max(1, rows/cols))*O      (O transposed back)
 *   packed_grads  bf16 bits, read only: device memory, or page-locked host memory with a
 *                 device mapping (cudaHostAlloc / cudaMallocHost, or cudaHostRegister with
 *                 a mapping), which the step's first pass then reads in place over the host
 *                 link, once, with no copy; pageable host memory is refused (NSM_ERR_ARG)
 *   packed_params device, fp32, updated in place (the owner's master copy)
 *   momentum      device, fp32, updated in place
 *   offsets       host, n int64 element offsets (shared by the three buffers)
 *   shapes        host, n {rows, cols}
 *   workspace     device, >= muon_workspace_bytes(shapes, n, ns_method, ns_steps)
 *                 bytes, 256-byte aligned; overwritten, except that its first 4n bytes
 *                 carry one exponent per matrix from one call to the next (below)
 *   stream        stream to launch on
 * Grads must not alias params or momentum.
 * Storage of X: the chain's input is held as U 2^k rounded once to the storage format,
 * k a per-matrix power of two, and s 2^-k (s = 1/(||U||_F + 1e-7)) multiplies the
 * products that read it; X is therefore s times U rounded to the format's significant
 * bits, with no range limit.  The norm is known only after the pass over U, so the step
 * stores U 2^k with the exponent the previous call on this table and workspace chose
 * (the first 4n bytes of the workspace) and makes a second pass over G and M only for
 * the matrices where that k put max|U| 2^k outside [2^4, 2^15): on the first call, or
 * after the gradients' magnitude jumps by a factor of about 16 or more.  Any content of
 * those bytes is safe.
 * Deterministic: identical inputs give bit-identical outputs whatever those bytes hold
 * (a power of two commutes with the rounding; only entries of U more than 2^18 below
 * their matrix's largest, which fp16 keeps as subnormals, can round differently), and a
 * matrix's result does not depend on the other matrices in the table. */
int muon_step(const void* packed_grads, float* packed_params, float* momentum,
              const int64_t* offsets, const int32_t* shapes, int n,
              float lr, float wd, float mu, int ns_method, int ns_steps, int nesterov,
              void* workspace, size_t workspace_bytes, nsm_stream_t stream);

/* muon_step that also writes the bf16 copy of every updated parameter into
 * params_bf16 (device, bf16, same offsets; NULL behaves like muon_step).  That copy is the
 * buffer an owner broadcasts to the other ranks and the next forward pass reads
 * ([DMZ] §两种packed buffer生命周期: the owner keeps the authoritative copy and broadcasts
 * the packed buffer); it is fused into the apply pass (2 more bytes per element).  It
 * must be 16-byte aligned and not overlap the other buffers. */
int muon_step_with_copy(const void* packed_grads, float* packed_params, float* momentum,
                        void* params_bf16, const int64_t* offsets, const int32_t* shapes, int n,
                        float lr, float wd, float mu, int ns_method, int ns_steps, int nesterov,
                        void* workspace, size_t workspace_bytes, nsm_stream_t stream);

/* Orthogonalisation only: out_i = NS(in_i / (||in_i||_F + 1e-7)) for every matrix of a
 * packed bf16 group (the same transpose rule and methods as muon_step).  in_bf16 and
 * out_bf16 are bf16 buffers sharing the offsets table, in device memory or in page-locked
 * host memory with a device mapping (then read or written in place over the host link);
 * they may not overlap, and pageable host memory is refused (NSM_ERR_ARG).
 * The input is held as in_i 2^k with k from a first pass over in_i (its sums and
 * largest entry), exact in the storage format for bf16 entries within 2^26 of the
 * largest.  Used to check and time the Newton-Schulz chain on its own. */
int muon_orthogonalize(const void* in_bf16, void* out_bf16,
                       const int64_t* offsets, const int32_t* shapes, int n,
                       int ns_method, int ns_steps,
                       void* workspace, size_t workspace_bytes, nsm_stream_t stream);

/* Orthogonalisation that allocates no device memory, for callers that cannot call
 * cudaMalloc: a host framework whose own caching pool owns every byte of device memory
 * (an allocation outside the pool can fail or fragment it), or a latency-critical loop
 * that cannot take the device synchronisation an allocation may imply.  It computes what
 * muon_orthogonalize computes, with the same kernels and bit-identical results, but keeps
 * its workspace and its launch plan in a 64 MiB array of device memory that is part of
 * the library itself (a file-scope __device__ array: every GPU that loads the library
 * holds it until the process exits).  The pages have no counterpart; this is a
 * convenience of the library.
 *   - Tables whose workspace and plan do not fit in the 64 MiB are rejected with
 *     NSM_ERR_WORKSPACE and nothing is launched (about 8M elements of square matrices
 *     fit; use muon_orthogonalize with a caller workspace for more).
 *   - Every call shares the array, which keeps the last call's contents.  Each call
 *     rewrites the workspace part before reading it, so nothing needs to start at zero;
 *     the plan part holds the last table's plan, which a call on the same table reuses
 *     without copying anything.  Calls that overlap on the GPU (two streams, or two host
 *     threads) race on the array: order them on one stream.
 *   - The first call on a device (and the first after its context was recreated, e.g.
 *     by a device reset) looks up the array's device address with cudaGetSymbolAddress,
 *     with that device current; make that first call before any stream capture.
 * Arguments are those of muon_orthogonalize without the workspace. */
int muon_orthogonalize_noalloc(const void* in_bf16, void* out_bf16,
                               const int64_t* offsets, const int32_t* shapes, int n,
                               int ns_method, int ns_steps, nsm_stream_t stream);

/* Fused AdamW step on one flat group ([DSM] §混合优化器的参数组构造: parameters without
 * use_muon go to AdamW; decoupled decay is the default mode):
 *     m <- b1*m + (1-b1)*g;  v <- b2*v + (1-b2)*g^2
 *     p <- p*(1 - lr*wd) - lr * (m/(1-b1^step)) / (sqrt(v/(1-b2^step)) + eps)
 *   grads bf16 (device, read only); params, exp_avg, exp_avg_sq fp32 (device, updated
 *   in place); numel >= 0 elements; step >= 1; all pointers 16-byte aligned. */
int adamw_step(const void* grads, float* params, float* exp_avg, float* exp_avg_sq,
               int64_t numel, float lr, float beta1, float beta2, float eps, float wd,
               int step, nsm_stream_t stream);

/* The tensor-core GEMM engine of the Newton-Schulz chain on one problem:
 *     out = alpha * A . op(B) + beta * aux + diag * I
 *   A      device, M x K row-major, row stride lda elements
 *   B      device; b_mn_major == 0: N x K row-major (op(B) = B^T, "K-major"),
 *          b_mn_major != 0: K x N row-major (op(B) = B, "MN-major"); row stride ldb
 *   out    device, M x N row-major, row stride ldo (written)
 *   aux    device, M x N row-major, row stride ldx, or NULL (then beta is ignored)
 *   fp16   0: every operand is bf16; 1: every operand is fp16.  fp32 accumulation.
 *   flags  NSM_GEMM_SYMMETRIC: the result is known to be symmetric (M == N and aux, if
 *          any, symmetric): only the tiles touching the upper triangle are computed and
 *          the strict upper triangle is mirrored into the lower one.
 *          NSM_GEMM_PAIR: run on the 2-SM kernel (clusters of two CTAs, 256 x 256 tiles)
 *          instead of the 1-CTA kernel (128 x 256 tiles).
 *   scratch device, >= nsm_gemm_scratch_bytes(M, N, flags) bytes, 128-byte aligned
 *          (holds the tensor maps and work list of the call)
 * Row strides must be multiples of 8 elements (>= the row length), pointers 16-byte
 * aligned, aux must not overlap out.  Exposed so the engine can be checked and timed
 * on its own; muon_step and muon_orthogonalize use the same kernel. */
#define NSM_GEMM_SYMMETRIC 1
#define NSM_GEMM_PAIR      2
int nsm_gemm(const void* a, int lda, const void* b, int ldb, void* out, int ldo,
             const void* aux, int ldx, int M, int N, int K, int b_mn_major, int fp16,
             int flags, float alpha, float beta, float diag, void* scratch,
             size_t scratch_bytes, nsm_stream_t stream);
size_t nsm_gemm_scratch_bytes(int M, int N, int flags);

/* Synchronises `stream`, then reads and clears the device status word that kernels set
 * when a bounded wait expires (or, in the checked build, when a bounds check fails).
 * *status_out = NSM_OK, NSM_ERR_TIMEOUT or NSM_ERR_BOUNDS.  Returns NSM_ERR_CUDA if the
 * synchronisation itself reports an error. */
int nsm_device_status(nsm_stream_t stream, int* status_out);

/* Where the first bounded wait that expired since the status word was last read gave up:
 * which kernel, which role inside the kernel and which barrier it was waiting on.
 * Every wait of the library's kernels is bounded (2 s of wall time); on expiry the
 * kernel records this, stops issuing work, lets its copies and MMAs in flight finish
 * and returns, so the context stays usable. */
#define NSM_KERNEL_GEMM       1  /* k_ns_gemm: the 1-CTA grouped GEMM */
#define NSM_KERNEL_GEMM_PAIR  2  /* k_ns_gemm_pair: the 2-SM grouped GEMM */
#define NSM_KERNEL_SMALL      3  /* k_ns_small: whole chains of matrices with m <= 128 */
#define NSM_KERNEL_SELFTEST   4  /* the kernels of nsm_status_selftest / nsm_bounds_selftest */
#define NSM_KERNEL_MOMENTUM   5  /* k_momentum_class, k_grad_norm (bounds checks only) */
#define NSM_KERNEL_TO_CLASS   6  /* k_to_class (bounds checks only) */
#define NSM_KERNEL_FROM_CLASS 7  /* k_from_class: apply or export (bounds checks only) */
#define NSM_KERNEL_ADAMW      8  /* k_adamw (bounds checks only) */
#define NSM_ROLE_PRODUCER     1  /* the thread issuing TMA loads */
#define NSM_ROLE_MMA          2  /* the thread issuing tensor-core MMAs */
#define NSM_ROLE_EPILOGUE     3  /* the epilogue warps draining TMEM */
#define NSM_ROLE_TEARDOWN     4  /* the end of the kernel: copies and MMAs still in flight */
#define NSM_SITE_STAGE_FULL   1  /* the TMA bytes of an operand stage */
#define NSM_SITE_STAGE_EMPTY  2  /* the MMAs that read an operand stage */
#define NSM_SITE_ACC_FULL     3  /* the MMAs of a TMEM accumulator */
#define NSM_SITE_ACC_EMPTY    4  /* the epilogue draining a TMEM accumulator */
#define NSM_SITE_DRAIN        5  /* the last MMAs before TMEM is freed */
#define NSM_SITE_SQUARE_FULL  6  /* the MMAs of an m x m product (k_ns_small) */
#define NSM_SITE_SQUARE_DONE  7  /* the epilogue writing an m x m iterate back (k_ns_small) */
#define NSM_SITE_XT_FULL      8  /* an X' chunk handed to the MMA thread (k_ns_small) */
#define NSM_SITE_XT_EMPTY     9  /* the MMA thread releasing an X' chunk (k_ns_small) */
#define NSM_SITE_STORES_DONE 10  /* the previous pass's X' stores landing (k_ns_small) */
#define NSM_SITE_SELFTEST    11  /* the self-test's barrier that nothing completes */
/* Sites of the checked build's bounds checks (status NSM_ERR_BOUNDS).  A TMA box is in
 * bounds when its first element lies inside the operand's matrix, its innermost
 * coordinate is a whole number of 16-byte units and its batch index is one of the
 * group's matrices; a plain access when every element it touches lies inside its
 * matrix (in the natural layout, the slot or the flat AdamW group), 16-byte vectors on
 * 16-byte boundaries. */
#define NSM_SITE_TMA_A          12  /* TMA load of the A operand (GEMM kernels) */
#define NSM_SITE_TMA_B          13  /* TMA load of the B operand (GEMM kernels) */
#define NSM_SITE_AUX            14  /* epilogue load of the aux operand (GEMM kernels) */
#define NSM_SITE_OUT            15  /* epilogue store of the output: TMA box or plain store */
#define NSM_SITE_TMA_X_LOAD     16  /* TMA load of an X chunk (k_ns_small) */
#define NSM_SITE_TMA_X_STORE    17  /* TMA store of an X' or O chunk (k_ns_small) */
#define NSM_SITE_NATURAL_LOAD   18  /* load from the packed natural layout (G, M, p) */
#define NSM_SITE_NATURAL_STORE  19  /* store to the packed natural layout (M, p, bf16 copy) */
#define NSM_SITE_SLOT_LOAD      20  /* load from a matrix's slot in the working layout */
#define NSM_SITE_SLOT_STORE     21  /* store to a matrix's slot in the working layout */
#define NSM_SITE_FLAT           22  /* AdamW's access to its flat group */
#define NSM_SITE_SELFTEST_BOUNDS 23 /* nsm_bounds_selftest's check of an index past its range */

/* nsm_device_status with the location: synchronises `stream`, reads and clears the
 * status word.  *status_out = NSM_OK, NSM_ERR_TIMEOUT or NSM_ERR_BOUNDS; then *kernel_out,
 * *role_out and *site_out are NSM_KERNEL_*, NSM_ROLE_* and NSM_SITE_* (0 with NSM_OK; the
 * self-test kernels and the elementwise kernels report role 0).  Only the first record
 * since the word was last read is kept.
 * Any of the three location pointers may be NULL. */
int nsm_device_status_detail(nsm_stream_t stream, int* status_out, int* kernel_out,
                             int* role_out, int* site_out);

/* Self-test of the bounded-wait status path: launches one CTA on `stream` whose bounded
 * wait on an mbarrier that nothing completes expires after wait_us microseconds (1 to
 * 2,000,000).  The kernel then records the timeout in the device status word, exactly as
 * a Newton-Schulz kernel that gave up would, and returns; the context stays usable.  The
 * next nsm_device_status reports NSM_ERR_TIMEOUT (and clears it).  Returns NSM_ERR_ARG,
 * with nothing launched, for wait_us out of range. */
int nsm_status_selftest(int wait_us, nsm_stream_t stream);

/* Self-test of the checked build's bounds checks: launches one thread on `stream` that
 * runs the bounds check the kernels use on the index one past the end of a one-element
 * range, and makes no access at all.  In the checked build (NSM_OPT_BOUNDS_CHECKS = 1)
 * the check fails and records NSM_ERR_BOUNDS with NSM_KERNEL_SELFTEST, role 0 and
 * NSM_SITE_SELFTEST_BOUNDS; in the regular build the checks are compiled out and nothing
 * is recorded.  Returns NSM_ERR_CUDA if the launch fails. */
int nsm_bounds_selftest(nsm_stream_t stream);

/* Host-to-device copy by the SMs, for uploading a step's inputs: `ctas` CTAs (0: 16) on
 * `stream` read `bytes` from page-locked host memory `src` (cudaHostAlloc /
 * cudaMallocHost, or registered with cudaHostRegister) through its device mapping, and
 * write them to device memory `dst`.  On the GB300 machines measured, 16 CTAs loading
 * over the host link sustained about 125-177 GB/s next to a running step, where the copy
 * engine's rate varied from about 40 to 207 GB/s, but they slowed the step itself by
 * 5-25%; with nothing else running both reach about 210 GB/s.  dst and src 16-byte aligned; any byte count.  Returns
 * NSM_ERR_NULL / NSM_ERR_ALIGN, NSM_ERR_ARG for ctas outside [0, 1024] or a src that is
 * not page-locked host memory with a device mapping (checked with cudaPointerGetAttributes
 * before anything is launched), NSM_ERR_CUDA if that query or the launch fails.  The
 * pages have no counterpart: it moves data only. */
int nsm_copy_to_device(void* dst, const void* src, size_t bytes, int ctas, nsm_stream_t stream);

/* Kernel timing for profiling.  While enabled, every kernel launch of muon_step,
 * muon_orthogonalize, adamw_step and nsm_gemm is bracketed by CUDA events on the
 * caller's stream.  nsm_timing_read_kind synchronises the recorded events and returns,
 * summed since the last reset for one kind of kernel: *ms (device time), *launches and
 * *work (the algorithmic work of those launches: flops for NSM_KIND_GEMM, bytes that
 * must cross HBM for the other kinds).  nsm_timing_read is the GEMM kind.  Any output
 * pointer may be NULL.  Not for use inside stream capture. */
#define NSM_KIND_GEMM      0  /* Newton-Schulz GEMM stages (tensor cores) */
#define NSM_KIND_MOMENTUM  1  /* the step's pass: momentum update, U 2^k into the working
                                  layout, per-tile sums of U^2 and largest |U| */
#define NSM_KIND_NORM      2  /* per-matrix norm, exponent and input factor */
#define NSM_KIND_LAYOUT    3  /* U 2^k into the working layout: the orthogonalisation's pass,
                                  and the step's second pass (work 0: it rewrites only the
                                  matrices whose exponent was out of range, usually none) */
#define NSM_KIND_APPLY     4  /* decay + apply (or the export of O) */
#define NSM_KIND_ADAMW     5  /* AdamW */
#define NSM_KIND_SMALL     6  /* whole Newton-Schulz chains of matrices with m <= 128 (bytes:
                                  every read and write of X; the kernel is HBM-bound) */
#define NSM_KIND_GRAD_NORM 7  /* the orthogonalisation's pass: sums of G^2, largest |G| */
int nsm_timing_enable(int enable);
int nsm_timing_read(double* gemm_ms, int64_t* gemm_launches, double* gemm_flops);
int nsm_timing_read_kind(int kind, double* ms, int64_t* launches, double* work);
int nsm_timing_reset(void);

/* Number of kernel launches the last successful muon_step / muon_orthogonalize /
 * adamw_step call made on this host thread. */
int nsm_last_launch_count(void);

/* Process-wide launch options.  They select between the library's own equivalent paths,
 * so that the paths can be compared with one another; every value gives the same
 * results.  A call made after a change uses the new value.  Values are 0 or 1 (0 to 2
 * for NSM_OPT_PDL); nsm_set_option returns NSM_ERR_ARG for an unknown option or value;
 * nsm_get_option returns the current value (NSM_ERR_ARG for an unknown option).  Not to
 * be changed while another host thread is inside a library call. */
#define NSM_OPT_PAIR_KERNELS 1  /* 1 (default): 2-SM GEMM kernel where it pays; 0: 1-CTA kernel only */
#define NSM_OPT_SMALL_KERNEL 2  /* 1 (default): chains of m <= 128 matrices in k_ns_small;
                                   0: those matrices go through the grouped launches */
#define NSM_OPT_PDL          3  /* 0: plain stream order; 1: programmatic dependent launch (a
                                   kernel's launch overlaps its predecessor's tail); 2 (default):
                                   auto, the latter for tables of at most 2^25 elements, where
                                   kernels are short enough for the launch latency to show */
#define NSM_OPT_BOUNDS_CHECKS 4 /* read only: 1 in the checked build (libnsmuon_checked.so),
                                   whose kernels check every global access and TMA box
                                   against its matrix before making it, record a failure
                                   (NSM_ERR_BOUNDS) and skip the access; 0 in the regular
                                   build.  nsm_set_option rejects it. */
#define NSM_OPT_SYM_STORAGE  5  /* 1 (default): where every grouped launch of a chain runs on the
                                   2-SM kernel, its symmetric m x m iterates are stored as their
                                   upper 256 x 256 tiles only, and a product reads a block below
                                   the diagonal from its mirror image; 0: every symmetric iterate
                                   is stored whole (each upper tile mirrored) */
int nsm_set_option(int option, int value);
int nsm_get_option(int option);

#ifdef __cplusplus
}
#endif

#endif /* NSMUON_H */
