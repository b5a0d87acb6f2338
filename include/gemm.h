/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense GEMM / GEMV library
 * (libdgemm_gb300.so).
 *
 * Operation (one call):
 *
 *     C <- act(alpha * op(A) @ op(B) + beta * C)
 *
 * op(A) is M x K, op(B) is K x N and C is M x N, following the BLAS naming of
 * "Matrix Multiplication Background User's Guide", section 2 (Math and Memory
 * Bounds); every output is a K-long dot product, 2*M*N*K floating-point
 * operations in all.  The guide's display formula for GEMM is lost in the
 * extracted text: the BLAS form above is the reading taken.  act is the
 * identity, LeakyReLU (the fused output transform of "OpenAI open-sources the
 * Triton GPU language (part 2)", section Matrix multiplication), ReLU, GELU
 * or SiLU.  Operands are bf16, fp16 or TF32 (fp32 words), products are
 * accumulated in fp32, C is fp32 or the operand type (gemm_run_ex: a separate
 * D, and a C of its own type).
 *
 * Storage is row-major ("Learning Triton One Kernel at a Time: Matrix
 * Multiplication", section Memory coalescing: a row is contiguous, a
 * transpose changes the strides, not the memory):
 *   transA = GEMM_OP_N: A is stored M x K,  op(A)(i,k) = A[i*lda + k]
 *   transA = GEMM_OP_T: A is stored K x M,  op(A)(i,k) = A[k*lda + i]
 *   transB = GEMM_OP_N: B is stored K x N,  op(B)(k,j) = B[k*ldb + j]
 *   transB = GEMM_OP_T: B is stored N x K,  op(B)(k,j) = B[j*ldb + k]
 *   C is stored M x N,                      C(i,j)     = C[i*ldc + j]
 * Leading dimensions count elements.  Entries of a row beyond its logical
 * width (the ld padding) are never read or written.
 *
 * Execution: gemm_run is asynchronous and stream-ordered on the caller's CUDA
 * stream; it returns after enqueueing its kernels.  All device pointers are
 * owned by the caller and must stay valid until the stream has run the call.
 * The plan owns its workspace (split-K partials, GEMV partials, the watchdog
 * word) and frees it in gemm_plan_destroy.  One plan must not be used by two
 * host threads, or on two streams whose work may overlap, at the same time.
 * The GEMM and GEMV kernels launch as programmatic dependents of the previous
 * kernel on the stream (CUDA programmatic dependent launch): their launch
 * and setup may overlap that kernel's last moments, but they touch no memory
 * before it has completed, so stream order holds as for a plain launch.  The
 * GEMM kernel lets its own dependents start early; a caller's kernel launched
 * after a gemm_run with the programmatic stream-serialization attribute must
 * therefore call cudaGridDependencySynchronize() (griddepcontrol.wait) before
 * it reads the result, as that attribute requires.  Set GEMM_PDL=0 in the
 * environment before gemm_plan_create for plain launches.
 *
 * Errors: argument problems are reported synchronously, before anything is
 * launched, as a gemm_status_t; nothing aborts or throws across this ABI.
 * There is no CPU fallback: without a usable sm_100-family GPU,
 * gemm_plan_create returns GEMM_ERR_NO_DEVICE.
 */
#ifndef DGEMM_GB300_GEMM_H
#define DGEMM_GB300_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct gemm_plan* gemm_plan_t;

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = 1,   /* null pointer, negative size, ld too small, bad enum  */
  GEMM_ERR_ALIGNMENT = 2,     /* pointer or leading dimension breaks the rules below */
  GEMM_ERR_UNSUPPORTED = 3,   /* size beyond what the kernels index (see gemm_run)   */
  GEMM_ERR_NO_DEVICE = 4,     /* no CUDA device, or not compute capability 10.x      */
  GEMM_ERR_OUT_OF_MEMORY = 5, /* workspace allocation failed                         */
  GEMM_ERR_CUDA = 6,          /* a CUDA runtime/driver call or a launch failed       */
  GEMM_ERR_TIMEOUT = 7,       /* a kernel's bounded wait ran out (watchdog)          */
  GEMM_ERR_DEBUG_CHECK = 8    /* debug build: a kernel's bounds or copy-rule check
                                 failed and the access was skipped (see below)    */
} gemm_status_t;

typedef enum { GEMM_OP_N = 0, GEMM_OP_T = 1 } gemm_op_t;

/* operand type _ C type */
typedef enum {
  GEMM_BF16_F32 = 0,
  GEMM_BF16_BF16 = 1,
  GEMM_F16_F32 = 2,
  GEMM_F16_F16 = 3,
  /* A and B are fp32 words read as TF32 by the tensor core: sign, exponent and
   * the 10 highest fraction bits (the 13 lowest are dropped), fp32
   * accumulation, C fp32 ("Matrix Multiplication Background User's Guide",
   * section 2.2, Table 1).  Every shape runs on the tensor cores, M = 1 or
   * N = 1 included.  Operands stored M/N-major (transA = T, transB = N) are
   * read by the MMAs where they are, except where the call is large enough
   * that copying one or both K-major into plan workspace first is estimated
   * faster (the in-place MMAs run ~10% longer with one such operand, ~44%
   * with both; a copy reads and writes the operand): 8192^3, for instance.
   * GEMM_TF32_TRANSPOSE=1 in the environment copies every M/N-major TF32
   * operand, =0 none (read at every call). */
  GEMM_TF32_F32 = 4
} gemm_dtype_t;

typedef enum {
  GEMM_ACT_NONE = 0,
  GEMM_ACT_LEAKY_RELU = 1, /* x < 0 ? slope*x : x  (the pages' example: "OpenAI open-sources the
                              Triton GPU language (part 2)", section Matrix multiplication) */
  GEMM_ACT_RELU = 2,       /* x < 0 ? 0 : x  (-0 and NaN pass unchanged)                    */
  GEMM_ACT_GELU = 3,       /* x * Phi(x), Phi the standard normal distribution function,
                              evaluated as erfc(-x / sqrt(2)) / 2 in fp32                    */
  GEMM_ACT_SILU = 4        /* x * sigmoid(x) = x / (1 + exp(-x)), in fp32                     */
} gemm_act_t;

/* The activation is applied in fp32 to alpha*acc + beta*C, before the
 * rounding to the output type; slope is read for GEMM_ACT_LEAKY_RELU only. */
typedef struct {
  int32_t act;
  float slope;
} gemm_epilogue_t;

/* Which kernels a call used. */
typedef enum {
  GEMM_PATH_NONE = 0,          /* M == 0 or N == 0: nothing launched                    */
  GEMM_PATH_TC = 1,            /* tcgen05 tensor-core GEMM, epilogue fused               */
  GEMM_PATH_TC_SPLITK = 2,     /* tcgen05 GEMM over K slices + fixed-order reduction     */
  GEMM_PATH_GEMV_ROWDOT = 3,   /* GEMV: one warp per contiguous row                      */
  GEMM_PATH_GEMV_COLSTREAM = 4,/* GEMV: threads own 8 contiguous columns, K split       */
  GEMM_PATH_GEMV_GENERIC = 5,  /* GEMV with strided operands (no 128-bit loads)          */
  GEMM_PATH_SCALE = 6,         /* K == 0 or alpha == 0: C <- act(beta*C)                 */
  GEMM_PATH_TC_SPLITK_CLUSTER = 7, /* tcgen05 GEMM, K in two halves on a cluster of two CTAs
                                  whose partial sums are added on chip: one launch, no
                                  workspace (the reduction of section 2.3 done in place) */
  GEMM_PATH_TC_TAIL_SPLIT = 8  /* tcgen05 GEMM: whole tiles for the full waves; only the
                                  tiles of the last, partly filled wave are split along K
                                  (section 3.2's tail wave), + reduction of those tiles  */
} gemm_path_t;

/* Plan decisions and the tile/wave quantization they imply ("Matrix
 * Multiplication Background User's Guide", section 3, Dimension Quantization
 * Effects: section 3.1 tile quantization, section 3.2 wave quantization). */
typedef struct {
  int32_t path;            /* gemm_path_t                                              */
  int32_t tile_m;          /* output tile rows (tensor-core paths)                     */
  int32_t tile_n;          /* output tile columns                                      */
  int32_t tile_k;          /* K elements per pipeline stage                            */
  int32_t cta_per_tile;    /* CTAs that work on one tile (1; 2 = a cluster of two: a    */
                           /* 256-row CTA pair, or the K halves of a split-K cluster)  */
  int32_t splitk;          /* K slices (1 = none)                                      */
  int32_t stages;          /* shared-memory pipeline depth                             */
  int32_t raster_group;    /* output-tile rows per rasterisation group                 */
  int32_t grid;            /* CTAs launched for the main kernel (gemm_choose_config:  */
                           /* 0 for the row-dot and generic GEMVs, whose grid comes   */
                           /* from the device's occupancy at launch)                  */
  int32_t sms;             /* streaming multiprocessors used for the wave size         */
  int64_t tiles;           /* output tiles = ceil(M/tile_m) * ceil(N/tile_n)           */
  int64_t units;           /* work units = tiles - tail_tiles + tail_tiles * splitk    */
                           /* (a 256-row pair tile is one unit of two CTAs; a K pair  */
                           /* tile is two units, its halves)                          */
  double waves;            /* units / wave size                                        */
  double tail_fraction;    /* (units mod wave) / wave: SMs busy in the last wave, 0=full */
  double useful_fraction;  /* M*N / (tiles*tile_m*tile_n): share of tile area in C     */
  int32_t launches;        /* kernels the call launched                                */
  int32_t tail_tiles;      /* tiles split along K and reduced by a second launch:      */
                           /* all tiles (split-K), the last wave's (tail split) or 0   */
  int64_t workspace_bytes; /* plan workspace the call used                             */
} gemm_config_info_t;

/* Create a plan bound to CUDA device `device` (the caller's current device is
 * restored before returning).  Queries the SM count and allocates the
 * watchdog word.  Returns GEMM_ERR_NO_DEVICE if the device does not exist or
 * is not compute capability 10.x, GEMM_ERR_INVALID_ARG if plan is NULL.
 * With GEMM_LOG=1 in the environment at creation, every successful gemm_run /
 * gemm_run_ex of the plan prints one line on stderr: the shape, the types and
 * the decisions of gemm_config_info_t (gemm_choose_config does the same).
 * With GEMM_NVTX=1 at creation, every gemm_run / gemm_run_ex of the plan is
 * an NVTX range ("gemm MxNxK types opA opB") on the calling thread, for a
 * profiler's timeline (no cost beyond the range calls; none without a tool). */
gemm_status_t gemm_plan_create(gemm_plan_t* plan, int device);

/* C <- act(alpha * op(A) @ op(B) + beta * C), enqueued on `stream` (a
 * cudaStream_t; NULL means the legacy default stream).  Calls may be captured
 * into a CUDA graph; a call whose shape, pointers and flags the plan has seen
 * before (same workspace size) adds only kernel launches to the capture.  See the top of this
 * file for the layout of A, B and C; all three are device pointers.
 *
 * Dispatch: M == 0 or N == 0 launches nothing; K == 0 or alpha == 0 gives
 * C <- act(beta*C) without reading A or B; M == 1 or N == 1 takes the
 * memory-bound GEMV kernels (no tensor cores: "Matrix Multiplication
 * Background User's Guide", section 2 notes that matrix-vector products are
 * always memory-bound); everything else takes the tcgen05 tensor-core kernel,
 * split along K when the output has too few tiles to fill the GPU (section
 * 2.3 mentions splitting along K followed by a reduction).  With beta == 0,
 * C is not read (NaN in C does not propagate).
 *
 * Rules, checked before any launch:
 *  - M, N, K >= 0 and each < 2^31; lda >= stored columns of A (K for N, M
 *    for T), ldb >= stored columns of B (N for N, K for T), ldc >= N; all >= 1.
 *  - A and B may be NULL only if M*N == 0 or K == 0 or alpha == 0; C may be
 *    NULL only if M*N == 0.
 *  - When A and B are read (M*N > 0, K > 0, alpha != 0), no byte of C (its
 *    M rows of N elements, ldc apart) may lie in A or B (their stored rows,
 *    lda / ldb apart).  Slices of one parent whose rows interleave without
 *    sharing a byte are accepted; with different leading dimensions and more
 *    than 2^20 rows on both sides, overlapping address ranges are rejected.
 *  - Every pointer is aligned to its element size.
 *  - Tensor-core path (M >= 2 and N >= 2): A, B and C are 16-byte aligned and
 *    lda, ldb, ldc times the element size are multiples of 16 bytes -- the
 *    rule of Table 1 of the guide's section 2.2 for FP16 (multiples of 8
 *    elements), which the Tensor Memory Accelerator requires here.
 *  - GEMM_TF32_F32 (always the tensor-core path): A and B 16-byte aligned with
 *    lda, ldb multiples of 4 elements (Table 1's TF32 row); C 4-byte aligned,
 *    and 16-byte aligned with ldc a multiple of 4 when N >= 4.
 * Violations return GEMM_ERR_INVALID_ARG or GEMM_ERR_ALIGNMENT.
 *
 * Split-K and GEMV with K split use the plan's workspace; the first call that
 * needs more than the plan holds grows it (stream-ordered allocation on
 * `stream`) and can return GEMM_ERR_OUT_OF_MEMORY.  Launch failures return
 * GEMM_ERR_CUDA.  A kernel whose bounded wait ran out sets the plan's
 * watchdog word (see gemm_plan_poll_error); the call itself still returns
 * GEMM_OK because it does not wait for the kernel.
 *
 * Results are deterministic: the same call on the same device gives the same
 * bits every time (split-K sums its slices in a fixed order). */
gemm_status_t gemm_run(gemm_plan_t plan, int64_t M, int64_t N, int64_t K,
                       const void* A, int64_t lda, const void* B, int64_t ldb,
                       void* C, int64_t ldc, float alpha, float beta,
                       gemm_dtype_t dtype, gemm_op_t transA, gemm_op_t transB,
                       gemm_epilogue_t epilogue, void* stream);

/* Free the plan and its workspace (synchronises the plan's device).  NULL is
 * accepted and ignored. */
gemm_status_t gemm_plan_destroy(gemm_plan_t plan);

/* Static, human-readable text for a status code. */
const char* gemm_status_string(gemm_status_t status);

/* Element types of gemm_run_ex's matrices. */
typedef enum { GEMM_TYPE_BF16 = 0, GEMM_TYPE_F16 = 1, GEMM_TYPE_F32 = 2,
               GEMM_TYPE_TF32 = 3 /* operands only (ab_type): fp32 words read as TF32 */ } gemm_type_t;

/* D <- act(alpha * op(A) @ op(B) + beta * C) with a separate output D: the
 * gemm_run operation where the C that beta scales is read from one matrix and
 * the result written to another, each with its own leading dimension and
 * element type (e.g. fp32 C in, bf16 D out).
 *   ab_type  GEMM_TYPE_BF16, GEMM_TYPE_F16 or GEMM_TYPE_TF32: A and B, as in gemm_run.
 *   d_type   GEMM_TYPE_F32 or ab_type (GEMM_TYPE_F32 with TF32 operands): D (M x N,
 *            row stride ldd >= N), held to
 *            gemm_run's rules for C (device pointer, alignment, NULL only
 *            if M*N == 0).
 *   c_type   GEMM_TYPE_BF16, GEMM_TYPE_F16 or GEMM_TYPE_F32: C (M x N, row
 *            stride ldc >= N), read only when beta != 0 (it may then be NULL
 *            and ldc is ignored); it needs only its element alignment.  C may
 *            be D itself (same pointer, ldc == ldd, c_type == d_type: that is
 *            gemm_run); otherwise the two must not share a byte.  C may
 *            overlap A or B (all three are only read); D may not.
 * Violations return GEMM_ERR_INVALID_ARG or GEMM_ERR_ALIGNMENT before any
 * launch.  Paths, workspace, streams and errors as in gemm_run; the plan's
 * last configuration is updated the same way.  The pages fuse input and
 * output transforms into the product ("OpenAI open-sources the Triton GPU
 * language (part 2)", section Matrix multiplication); a separate D is the
 * output side of that with C left intact. */
gemm_status_t gemm_run_ex(gemm_plan_t plan, int64_t M, int64_t N, int64_t K, const void* A,
                          int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc,
                          gemm_type_t c_type, void* D, int64_t ldd, gemm_type_t d_type, float alpha,
                          float beta, gemm_type_t ab_type, gemm_op_t transA, gemm_op_t transB,
                          gemm_epilogue_t epilogue, void* stream);

/* Decisions of the plan's most recent gemm_run (path, tile, split-K, grid,
 * waves, tail fraction, kernels launched).  GEMM_ERR_INVALID_ARG on NULL. */
gemm_status_t gemm_plan_last_config(gemm_plan_t plan, gemm_config_info_t* out);

/* Wait for `stream`, then read and clear the plan's watchdog word: returns
 * GEMM_ERR_TIMEOUT if any kernel of this plan gave up on a bounded wait since
 * the last poll, GEMM_ERR_DEBUG_CHECK if (debug build) a device-side check
 * failed, GEMM_OK otherwise, GEMM_ERR_CUDA if the stream failed. */
gemm_status_t gemm_plan_poll_error(gemm_plan_t plan, void* stream);

/* The word the last gemm_plan_poll_error read, before it was cleared (0:
 * nothing happened).  Bits 0-15: the bounded waits that ran out (producer,
 * MMA, epilogue, exchange, ...); bit 30: a debug-build check failed, and bit
 * 16 + s for each failing site s: 0 a TMA copy's coordinates (innermost
 * coordinate times the element size not a multiple of 16 bytes, or a store
 * starting at a negative coordinate), 1 an epilogue store, 2 an epilogue load
 * of the C that beta scales, 3 the in-kernel split-K reduction, 4 the tile
 * reduction kernel, 5 a GEMV kernel, 6 the K == 0 / alpha == 0 kernel, 7 the
 * TF32 operand transpose.  GEMM_ERR_INVALID_ARG on NULL. */
gemm_status_t gemm_plan_last_error_bits(gemm_plan_t plan, int64_t* bits);

/* 1 in the debug build of the library (libdgemm_gb300_debug.so, compiled
 * with DG_DEBUG), 0 in the release build.  The debug build checks, on the
 * device, every plain global load and store of every kernel against the
 * byte ranges of the call's own buffers (operands, output, the C that beta
 * scales, plan workspace and counters; a GEMV matrix row or a column strip
 * as a whole) and every TMA copy's coordinates against the copy rules,
 * before the access; a failed check skips the access (no trap, no fault)
 * and sets the plan's error word, which gemm_plan_poll_error reports as
 * GEMM_ERR_DEBUG_CHECK.  A skipped TMA load leaves its barrier incomplete,
 * so the bounded waits behind it run out as well.  gemm_gemv_noalloc has no
 * plan to report through and is not checked.  For its own tests the debug
 * build reads GEMM_DEBUG_SHRINK=n once per process: the output's byte
 * range is taken n bytes shorter than it is, so that the checks of the last
 * output elements fail while every access stays inside the buffer. */
int gemm_debug_build(void);

/* Limit, in nanoseconds, of every bounded wait inside this plan's kernels
 * (default 2e9; the environment variable GEMM_WATCHDOG_NS overrides the
 * default at plan creation).  Values < 1000 are rejected. */
gemm_status_t gemm_plan_set_watchdog(gemm_plan_t plan, uint64_t timeout_ns);

/* Benchmark mode ("Matrix Multiplication Background User's Guide", section
 * 2.3: some frameworks time every implementation option once, before the
 * real work, and keep the fastest).  With enable != 0, the first
 * tensor-core gemm_run of each (M, N, K, lda, ldb, ldc, dtype, transA,
 * transB, beta != 0) on this plan times the planner's leading candidates
 * (its pick and up to five more estimated within 15% of the best): one
 * warm-up and three timed runs each, on the call's stream, writing into a
 * scratch copy of C (stream-ordered allocation the size of C; C, A and B
 * are not modified).  The fastest is kept for every later call of that
 * shape on this plan, whatever the pointers.  That first call blocks the
 * host until the trials have run (a one-time cost per shape); if anything
 * fails the planner's pick is kept.  enable = 0 (the default; the
 * environment variable GEMM_AUTOTUNE=1 turns it on at plan creation)
 * uses the planner's estimate alone.  Not applied while `stream` is being
 * captured into a CUDA graph (the planner's estimate decides there).
 * Ignored while any GEMM_FORCE_* /
 * GEMM_RASTER_GROUP / GEMM_SPLITK_CLUSTER / GEMM_TAIL_SPLIT override is set.
 * GEMM_ERR_INVALID_ARG on NULL. */
gemm_status_t gemm_plan_set_autotune(gemm_plan_t plan, int enable);

/* Number of shapes benchmark mode has timed on this plan (bounded: the
 * record is cleared past 4096 shapes).  GEMM_ERR_INVALID_ARG on NULL. */
gemm_status_t gemm_plan_tuned_count(gemm_plan_t plan, int64_t* count);

/* Watchdog self-test: launch one CTA that waits on a barrier nothing will
 * ever arrive on, with this plan's limit, then wait for `stream`.  Returns
 * GEMM_ERR_TIMEOUT when the wait ran out and the kernel returned on its own
 * (the expected result; the context stays usable), GEMM_OK if it did not. */
gemm_status_t gemm_plan_selftest_watchdog(gemm_plan_t plan, void* stream);

/* The argument checks of gemm_run without a plan or a device: returns the
 * status gemm_run would return before launching anything. */
gemm_status_t gemm_check_args(int64_t M, int64_t N, int64_t K,
                              const void* A, int64_t lda, const void* B, int64_t ldb,
                              const void* C, int64_t ldc, float alpha,
                              gemm_dtype_t dtype, gemm_op_t transA, gemm_op_t transB,
                              gemm_epilogue_t epilogue);

/* The argument checks of gemm_run_ex without a plan or a device. */
gemm_status_t gemm_check_args_ex(int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                                 const void* B, int64_t ldb, const void* C, int64_t ldc,
                                 gemm_type_t c_type, const void* D, int64_t ldd, gemm_type_t d_type,
                                 float alpha, float beta, gemm_type_t ab_type, gemm_op_t transA,
                                 gemm_op_t transB, gemm_epilogue_t epilogue);

/* The planner of gemm_run as a pure host function: the decisions it would
 * make for this problem on a GPU with `sms` multiprocessors.  Does not need a
 * device.  Honours the GEMM_FORCE_TILE / GEMM_FORCE_SPLITK overrides.
 * `launches` counts the GEMM's own kernels: with TF32 operands stored
 * M/N-major, gemm_run may launch a K-major copy of one or both first (see
 * GEMM_TF32_F32), which its own record (gemm_plan_last_config) counts. */
gemm_status_t gemm_choose_config(int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                                 gemm_op_t transA, gemm_op_t transB, int32_t sms,
                                 gemm_config_info_t* out);

/* Tile and wave quantization of an M x N output cut into tile_m x tile_n
 * tiles, each split into `splitk` K slices, on `sms` multiprocessors running
 * `ctas_per_sm` tiles at a time ("Matrix Multiplication Background User's
 * Guide", sections 3.1 and 3.2).  Fills tiles, units, waves, tail_fraction,
 * useful_fraction, tile_m, tile_n, splitk and sms.  Pure host arithmetic. */
gemm_status_t gemm_quantization(int64_t M, int64_t N, int32_t tile_m, int32_t tile_n,
                                int32_t splitk, int32_t sms, int32_t ctas_per_sm,
                                gemm_config_info_t* out);

/* GEMV that allocates nothing.  The pages have no counterpart: this entry
 * point exists for callers that may not call cudaMalloc where they run a
 * GEMV -- a plugin inside a framework or inference server that owns all
 * device memory through its own pool allocator, or a latency-critical loop
 * that cannot take cudaMalloc's implicit device synchronisation -- and so
 * cannot create a plan (gemm_plan_create allocates) or let one grow.
 *
 * Same arguments as gemm_run, without the plan; same results as gemm_run for
 * the shapes it accepts: the column-stream GEMV, i.e. M == 1 with B stored
 * K x N (transB = GEMM_OP_N) and N >= 2, or N == 1 with A stored K x M
 * (transA = GEMM_OP_T); K >= 1, alpha != 0; the matrix operand 16-byte
 * aligned with ld * 2 a multiple of 16 bytes.  Other shapes, and outputs
 * longer than 2,097,152 elements (the fixed scratch), return
 * GEMM_ERR_UNSUPPORTED before anything is launched; argument errors are
 * those of gemm_run.
 *
 * Runs on the calling thread's current device; `stream` must belong to it.
 * Its scratch is a fixed 4 MiB device array of the library; the call zeroes
 * the part that must start at zero.  CUDA loads the library's device code
 * lazily: the first call on a device looks up that array's address
 * (cudaGetSymbolAddress), which loads it there and takes its 4 MiB from the
 * device's free memory until the process exits (GEMM_ERR_OUT_OF_MEMORY if no
 * room is left).  Make that first call before a pool allocator reserves the
 * device's memory, and before any stream capture; later calls allocate
 * nothing.  All calls on a device share the array: calls whose kernels may
 * overlap on the GPU race and must be ordered by the caller (one stream, or
 * events).  No cudaMalloc, cudaFree or other allocating call is made. */
gemm_status_t gemm_gemv_noalloc(int64_t M, int64_t N, int64_t K,
                                const void* A, int64_t lda, const void* B, int64_t ldb,
                                void* C, int64_t ldc, float alpha, float beta,
                                gemm_dtype_t dtype, gemm_op_t transA, gemm_op_t transB,
                                gemm_epilogue_t epilogue, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DGEMM_GB300_GEMM_H */
