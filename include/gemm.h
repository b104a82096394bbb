/*
 * gemm.h -- C ABI of the GB300 (sm_103a) blocked matrix-multiply library.
 *
 * The library computes the blocked matrix multiply of "Chapter 13: The Blocked
 * Matmul Kernel" (section 13.1, Worked Example 13.1.1):
 *
 *     C[M,N] = A[M,K] @ B[K,N],
 *
 * as a 2D grid of output tiles, each accumulating its K-loop of partial
 * products into an fp32 accumulator initialised once (section 13.1, the
 * "common trap" on where the accumulator is initialised), with every
 * out-of-range M, N and K element contributing exactly zero (section 13.2,
 * three-way masking; "Triton from zero, Lesson 4: Block Pointers", section 3,
 * zero padding), the result rounded once to the output type at the store
 * (section 13.3), and an explicit choice between tf32 and exact fp32 for fp32
 * inputs ("Triton matmul", the "Precision" section).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Pointers A, B, C are DEVICE pointers owned by the caller; the library never
 * frees or retains them past the call. Leading dimensions are in ELEMENTS.
 *   A: M x K; GEMM_ROW_MAJOR -> A[i,k] at A + i*lda + k (lda >= K);
 *             GEMM_COL_MAJOR -> A[i,k] at A + k*lda + i (lda >= M).
 *   B: K x N; GEMM_ROW_MAJOR -> B[k,j] at B + k*ldb + j (ldb >= N);
 *             GEMM_COL_MAJOR -> B[k,j] at B + j*ldb + k (ldb >= K)
 *             (the [N,K] storage of the transposed-B read of "Triton from
 *             zero, Lesson 4", homework 2).
 *   C: M x N, always row-major: C[i,j] at C + i*ldc + j (ldc >= N).
 * Only C[i,j] with i < M and j < N is written; bytes of C outside that set
 * (row tails when ldc > N) are left untouched. A and B are read only inside
 * their logical extents.
 *
 * Arithmetic: products are accumulated in fp32 and rounded once to out_dtype
 * with round-to-nearest-even. K == 0 writes zeros (the empty sum). M == 0 or
 * N == 0 is a no-op returning GEMM_OK.
 *
 * Precision (fp32 inputs only): GEMM_PREC_DEFAULT means GEMM_PREC_EXACT_FP32;
 * GEMM_PREC_TF32 runs the tensor cores on tf32 operands (the low 13 mantissa bits
 * of each fp32 input are ignored; max |err| <= 2e-3 * sum_k |a_ik b_kj|), reading
 * row- and column-major operands alike in place (a product with a short K that the
 * planner gives to the fp32 FMA kernel, see gemm_run_ex, is computed in full fp32).
 * GEMM_PREC_EXACT_FP32 keeps fp32 accuracy (max |err| <= 1e-6 * sum_k |a_ik b_kj|
 * on the library's tests): each operand is split into two tf32 parts and the
 * three significant partial products run on the tensor cores, accumulating in
 * fp32 (tiny problems use fp32 fused multiply-adds). 16-bit inputs accept
 * GEMM_PREC_DEFAULT (fp32 accumulator) and, for fp16 inputs only,
 * GEMM_PREC_F16_ACC: the fp16 accumulator of "Chapter 13: The Blocked Matmul
 * Kernel", section 13.3 (Worked Example 13.3.1), kept to show what it costs. The
 * running total is an fp16 value that starts at +0; for every chunk of
 * GEMM_OPT_ACC_CHUNK consecutive K indices (from k = 0; default 16) the chunk's dot
 * product is formed in fp32, rounded to fp16, and added to the running total with
 * an fp16 round-to-nearest-even add; the total is then converted to out_dtype.
 * Chunks that are multiples of 16 run on the tensor cores (each chunk's fp32 dot is
 * one or more tcgen05.mma.kind::f16 into a fresh TMEM accumulator); other
 * multiples of 8 (the pages' BLOCK_K = 8) run on fp32 fused multiply-adds.
 *
 * Errors: checks on the host return a status and launch nothing. Work is
 * asynchronous on the given stream, so a GEMM_OK return means "launched";
 * faults found by the device (a bounded wait that expired) are reported by
 * gemm_get_status. A misaligned pointer or leading dimension is not an error:
 * the library stages such an operand through an aligned workspace that the
 * handle owns.
 *
 * Threads and streams: a handle may be used from one host thread at a time.
 * Its device buffers (staged operands, split-K partials, flags and epoch) are
 * reused by every call, so the calls made on one handle must run one after
 * another on the GPU: one stream, or streams ordered by events. Work that runs
 * concurrently takes one handle per stream. (gemm_run_host orders its own
 * internal streams.)
 */
#ifndef GEMM_GB300_H
#define GEMM_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

typedef struct gemm_handle_s *gemm_handle_t;

typedef enum { GEMM_F32 = 0, GEMM_F16 = 1, GEMM_BF16 = 2 } gemm_dtype_t;

typedef enum {
  GEMM_PREC_DEFAULT = 0,   /* exact fp32 for fp32 inputs; the only mode for 16-bit inputs */
  GEMM_PREC_TF32 = 1,      /* fp32 inputs on the tf32 tensor-core path */
  GEMM_PREC_EXACT_FP32 = 2, /* fp32 inputs at fp32 accuracy (split-tf32 tensor cores) */
  GEMM_PREC_F16_ACC = 3     /* fp16 inputs, fp16 accumulator rounded every K-chunk */
} gemm_precision_t;

typedef enum { GEMM_ROW_MAJOR = 0, GEMM_COL_MAJOR = 1 } gemm_layout_t;

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = 1, /* null/negative/overlapping/too-small argument */
  GEMM_ERR_UNSUPPORTED = 2, /* a valid request this library does not implement */
  GEMM_ERR_ALIGNMENT = 3,   /* a pointer not aligned to its element size */
  GEMM_ERR_NO_MEMORY = 4,   /* workspace allocation failed */
  GEMM_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed */
  GEMM_ERR_TIMEOUT = 6,     /* a device-side bounded wait expired (see gemm_get_status) */
  GEMM_ERR_DEVICE = 7       /* no usable sm_103 device */
} gemm_status_t;

/* Create a handle bound to CUDA device `device`. On success *out receives the
 * handle (free it with gemm_destroy). Allocates the device status word.
 * Errors: INVALID_ARG (out == NULL), DEVICE (no such device or not sm_103),
 * CUDA, NO_MEMORY. */
GEMM_API gemm_status_t gemm_create(gemm_handle_t *out, int device);

/* Free the handle, its workspace and its status word. Synchronises the device
 * first so no launched work still uses the workspace. NULL is a no-op. */
GEMM_API void gemm_destroy(gemm_handle_t h);

/* C = A @ B with row-major A and B on the legacy default stream.
 * Same as gemm_run_ex(..., GEMM_ROW_MAJOR, GEMM_ROW_MAJOR, NULL). */
GEMM_API gemm_status_t gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                const void *A, int64_t lda, const void *B, int64_t ldb,
                                void *C, int64_t ldc, gemm_dtype_t in_dtype,
                                gemm_dtype_t out_dtype, gemm_precision_t precision_mode);

/* C = A @ B with explicit operand layouts, enqueued on `cuda_stream` (a
 * cudaStream_t; NULL = legacy default stream). The host-side planner picks the
 * kernel -- the tcgen05 tensor-core kernels for 16-bit inputs and tf32 mode; for exact
 * fp32, the tensor cores on operands split once into tf32 hi and lo parts (three tf32
 * products, K summed in 128-long chunks in fp32 registers), or the fp32 FMA kernel for
 * problems too small to fill the tensor-core tiles; and the FMA kernel, for any input
 * dtype, for a K of at most 24 with at most 2^22 outputs unless one of the tile options
 * (GEMM_OPT_CTA_PAIR, BLOCK_N, STAGE_K, TILE_ROWS) is set -- stages misaligned operands,
 * and launches.
 * Errors (nothing launched): INVALID_ARG for h == NULL, negative sizes, a null
 * pointer with a non-empty extent, a leading dimension below its minimum, an
 * unknown enum, or C's span overlapping A's or B's; UNSUPPORTED for a
 * precision other than DEFAULT with 16-bit inputs; ALIGNMENT for a pointer not
 * aligned to its element size; NO_MEMORY/CUDA from staging or launch. */
GEMM_API gemm_status_t gemm_run_ex(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                   const void *A, int64_t lda, const void *B, int64_t ldb,
                                   void *C, int64_t ldc, gemm_dtype_t in_dtype,
                                   gemm_dtype_t out_dtype, gemm_precision_t precision_mode,
                                   gemm_layout_t a_layout, gemm_layout_t b_layout,
                                   void *cuda_stream);

/* C = A @ B for operands in HOST memory (A, B, C are host pointers; pinned memory makes
 * the copies asynchronous and fast, pageable memory works but copies synchronously).
 * Same arguments, layouts and checks as gemm_run_ex. The handle copies row panels of A and
 * column panels of B to the device in turn on its own streams; each arriving panel
 * completes a block of C (its rows or columns against every panel of the other operand
 * already there), which is multiplied and copied back while later panels copy in. The work
 * starts after everything enqueued on `cuda_stream` before the call, and `cuda_stream`
 * waits for its end (C is complete in host memory once that stream reaches this point).
 * The device copies live in a handle-owned buffer that grows on demand (growing it waits
 * for the handle's earlier host-path calls). Device-side faults are reported by
 * gemm_get_status. */
GEMM_API gemm_status_t gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                     const void *A, int64_t lda, const void *B, int64_t ldb,
                                     void *C, int64_t ldc, gemm_dtype_t in_dtype,
                                     gemm_dtype_t out_dtype, gemm_precision_t precision_mode,
                                     gemm_layout_t a_layout, gemm_layout_t b_layout,
                                     void *cuda_stream);

/* Synchronise `cuda_stream` (NULL = legacy default stream), then read and clear
 * the handle's device status word. Returns GEMM_OK, GEMM_ERR_TIMEOUT when a
 * kernel's bounded wait expired since the last call (its C is then
 * undefined), or GEMM_ERR_CUDA when the synchronisation itself failed. */
GEMM_API gemm_status_t gemm_get_status(gemm_handle_t h, void *cuda_stream);

/* Static description of a status code; never NULL. */
GEMM_API const char *gemm_strerror(gemm_status_t s);

/* ---------------------------------------------------------------- tuning */

typedef enum {
  GEMM_OPT_WAIT_TIMEOUT_US = 0, /* device bounded-wait limit in microseconds (default 2000000) */
  GEMM_OPT_FORCE_PATH = 1,      /* 0 auto, 1 tensor cores, 2 fp32 FMA kernel (any input dtype) */
  GEMM_OPT_GROUP_M = 2,         /* tile rows per raster group of the persistent schedule (>= 1) */
  GEMM_OPT_MAX_CTAS = 3,        /* cap on persistent CTAs (0 = one per SM) */
  GEMM_OPT_FAULT_STALL_PRODUCER = 4, /* test hook: 1 = the tensor-core kernel's loader issues
                                        nothing, so the consumers' bounded waits expire and the
                                        kernel reports GEMM_ERR_TIMEOUT; v >= 2 = the loader of
                                        CTA rank (v & 1) of a pair (the single CTA's loader)
                                        stops after v >> 1 stage fills, with copies still in
                                        flight; 0 = off */
  GEMM_OPT_FORCE_STAGING = 5,   /* 1 = stage A and B through the workspace even when aligned */
  GEMM_OPT_CTA_PAIR = 6,        /* tensor-core tiles: 0 auto, 1 single-CTA (128 rows),
                                   2 CTA-pair (256 rows, cta_group::2 on two SMs) */
  GEMM_OPT_BLOCK_N = 7,         /* tensor-core tile width: 0 auto, 128 or 256 */
  GEMM_OPT_EXACT_CHUNK = 8,     /* exact fp32: 32-long K-blocks summed in TMEM before each
                                   fp32 register add (0 = by K: k_blocks/24 in [1, 16]; 1..64) */
  GEMM_OPT_STREAM_K = 9,        /* split the last, partly filled rounds of tiles along K
                                   (fixed-order reduction, handle-owned workspace):
                                   0 when it pays (>= 2 whole rounds first, >= 64 K-blocks),
                                   1 never, 2 whenever the schedule allows */
  GEMM_OPT_HOST_PANEL = 10,     /* gemm_run_host: rows of A and columns of B per pipelined
                                   copy panel, a multiple of 256 (0 = auto: about 1/6 of the
                                   extent, >= 1024; widened to keep <= 24 such panels); the
                                   last two panels' worth is cut in halves down to 256 */
  GEMM_OPT_ACC_CHUNK = 11,      /* GEMM_PREC_F16_ACC: K indices per fp16 rounding of the
                                   running total, a multiple of 8 (0 = default 16) */
  GEMM_OPT_STAGE_K = 12,        /* 128-byte K-blocks per pipeline stage of the CTA-pair
                                   kernel: 0 auto, 1, or 2 (K-major 16-bit operands only;
                                   otherwise GEMM_ERR_UNSUPPORTED at run time) */
  GEMM_OPT_TILE_ROWS = 13,      /* rows of A per CTA of the CTA-pair kernel (its tile has
                                   twice as many): 0 = 128, or a multiple of 8 in [64, 128]
                                   (K-major A and the fp32 accumulator only; otherwise
                                   GEMM_ERR_UNSUPPORTED at run time) */
  GEMM_OPT_TF32_TRANSPOSE = 14  /* tf32 mode, an MN-major fp32 operand (row-major B,
                                   column-major A): 0 = the tensor cores read it in place
                                   (128-byte swizzle with 32-byte atoms), 1 = copy it
                                   transposed into K-major form first */
} gemm_option_t;

/* Set a per-handle option; INVALID_ARG for an unknown option or bad value. */
GEMM_API gemm_status_t gemm_set_option(gemm_handle_t h, gemm_option_t opt, int64_t value);

/* Number of kernels this handle has launched since it was created. */
GEMM_API gemm_status_t gemm_get_launch_count(gemm_handle_t h, uint64_t *count);

/* Timing hook for the main kernel of a product. With start_event and end_event both
 * cudaEvent_t handles (created by the caller, on this handle's device), every later
 * gemm_run / gemm_run_ex / gemm_run_strided call on this handle records start_event on
 * its stream immediately before it launches the GEMM kernel itself -- after any staging
 * copies (misaligned operands, transposed copies under GEMM_OPT_TF32_TRANSPOSE or for the
 * fp16 accumulator, the hi/lo split of exact fp32)
 * -- and end_event immediately after it, so that the caller can time that kernel apart
 * from the copies with cudaEventElapsedTime. Both NULL turns the hook off (the default).
 * The events stay owned by the caller, who must keep them alive while the hook is set.
 * Errors: INVALID_ARG for h == NULL or exactly one of the two events NULL. */
GEMM_API gemm_status_t gemm_set_kernel_events(gemm_handle_t h, void *start_event,
                                              void *end_event);

/* ------------------------------------------------------------- planning */

typedef enum {
  GEMM_PATH_NONE = 0,      /* nothing to do (M == 0 or N == 0) */
  GEMM_PATH_ZERO_FILL = 1, /* K == 0: C is set to zero */
  GEMM_PATH_TCGEN05 = 2,   /* TMA + mbarrier pipeline + tcgen05.mma, TMEM accumulator */
  GEMM_PATH_FMA = 3,       /* fp32 fused multiply-add tiles (tiny exact fp32, short K) */
  GEMM_PATH_TCGEN05_3XTF32 = 4, /* exact fp32 on the tensor cores: operands split into tf32
                                   hi/lo parts, three products in one fp32 accumulator */
  GEMM_PATH_TCGEN05_F16ACC = 5   /* fp16 accumulator on the tensor cores: each K-chunk's
                                   fp32 dot from TMEM is rounded into an fp16 running total */
} gemm_path_t;

typedef struct {
  int32_t path;           /* gemm_path_t */
  int32_t tile_m, tile_n, tile_k; /* output tile and K-chunk, in elements */
  int64_t grid_m, grid_n; /* output tiles along M and N */
  int64_t k_iters;        /* K-chunks per tile: ceil(K / tile_k) */
  int32_t stages;         /* shared-memory pipeline depth (tensor-core path) */
  int32_t stage_a, stage_b; /* 1 if the operand is copied to an aligned workspace first */
  int32_t a_mn_major, b_mn_major; /* operand read M/N-major (1) or K-major (0) */
  int32_t tma_store;      /* 1 if the epilogue writes C with TMA stores */
  int64_t ctas;           /* CTAs launched (persistent schedule; pairs count twice) */
  int64_t workspace_bytes; /* workspace the call needs */
  int32_t cta_pair;       /* 1 if tiles run on CTA pairs (two SMs per tile) */
  int32_t split_tiles;    /* tiles of the last rounds split along K (split-K) */
} gemm_plan_info_t;

/* Host-only: the plan gemm_run_ex would use for these arguments on a GPU with
 * `sm_count` SMs, without touching any device. Same argument checks and
 * return codes as gemm_run_ex; h may be NULL (default options). */
GEMM_API gemm_status_t gemm_plan(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                 const void *A, int64_t lda, const void *B, int64_t ldb,
                                 void *C, int64_t ldc, gemm_dtype_t in_dtype,
                                 gemm_dtype_t out_dtype, gemm_precision_t precision_mode,
                                 gemm_layout_t a_layout, gemm_layout_t b_layout,
                                 int32_t sm_count, gemm_plan_info_t *info);

/* ------------------------------------------------------------- row softmax */

/* Row softmax, the second workload of the pages ("Triton from zero, Lesson 4: Block
 * Pointers", homework 4): for each of the M rows of the row-major matrix X (leading
 * dimension ldx >= N, in elements),
 *     Y[i, j] = exp(X[i, j] - m_i) / sum_k exp(X[i, k] - m_i),   m_i = max_k X[i, k],
 * over the row's N values only (the homework's -inf padding of a tile's extra columns adds
 * nothing). Y is row-major with ldy >= N; bytes of Y past column N are untouched. In
 * place (Y == X, ldy == ldx, same dtype) is allowed; other overlaps are
 * GEMM_ERR_INVALID_ARG. Arithmetic in fp32; in_dtype and out_dtype any of the three. A row
 * holding a NaN or +inf, or only -inf, gives NaN (as the formula does). M == 0 or N == 0
 * is a no-op. Asynchronous on `cuda_stream`. */
GEMM_API gemm_status_t gemm_softmax_rows(gemm_handle_t h, int64_t M, int64_t N, const void *X,
                                         int64_t ldx, void *Y, int64_t ldy, gemm_dtype_t in_dtype,
                                         gemm_dtype_t out_dtype, void *cuda_stream);

/* ------------------------------------------------------------------- tuning */

typedef struct {
  int32_t cta_pair;   /* GEMM_OPT_CTA_PAIR value of the choice (1 single-CTA, 2 pairs) */
  int32_t block_n;    /* GEMM_OPT_BLOCK_N value (128 or 256) */
  int32_t stream_k;   /* GEMM_OPT_STREAM_K value (0 auto, 1 never, 2 when possible) */
  int32_t stage_k;    /* GEMM_OPT_STAGE_K value (1 or 2) */
  int32_t group_m;    /* GEMM_OPT_GROUP_M value */
  int32_t tile_rows;  /* GEMM_OPT_TILE_ROWS value (128 for single-CTA tiles) */
  int32_t candidates; /* configurations timed */
  float best_us;      /* mean time per product of the choice, microseconds */
  float default_us;   /* the same for the untuned plan (the first candidate) */
} gemm_tune_result_t;

/* Times the tensor-core configurations this problem admits -- tile shape (single-CTA or
 * CTA-pair rows, 128 or 256 columns), split-K of the last rounds, one or two K-blocks per
 * pipeline stage, raster group height -- `iters` runs each after one warm-up, on
 * `cuda_stream`, and keeps the fastest for the problem's signature (M, N, K, dtypes,
 * precision, layouts): later calls on this handle with that signature (gemm_run,
 * gemm_run_ex, gemm_plan, and the products inside gemm_run_strided and gemm_run_host)
 * use it in place of the handle's own values of those six options. The untuned plan is
 * one of the candidates, so the choice is never slower as measured. Blocking: returns
 * after the last timing. It runs the real product, so C is written (with the product).
 * Problems that do not take the plain tensor-core path (exact fp32, the fp16 accumulator,
 * short-K, tiny or K = 0 problems) have a single candidate. `iters` in [1, 1000]. Different
 * choices sum in different orders: results stay within the precision bounds but may
 * differ in the last bits from the untuned plan. `result` may be NULL. */
GEMM_API gemm_status_t gemm_tune(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void *A,
                                 int64_t lda, const void *B, int64_t ldb, void *C, int64_t ldc,
                                 gemm_dtype_t in_dtype, gemm_dtype_t out_dtype,
                                 gemm_precision_t precision_mode, gemm_layout_t a_layout,
                                 gemm_layout_t b_layout, void *cuda_stream, int32_t iters,
                                 gemm_tune_result_t *result);

/* Forgets every choice gemm_tune made on this handle. */
GEMM_API gemm_status_t gemm_tune_clear(gemm_handle_t h);

/* ------------------------------------------------------- six-stride interface */

/* C = A @ B for any 2D views: element (i, k) of A is at A + i * stride_am + k * stride_ak,
 * (k, j) of B at B + k * stride_bk + j * stride_bn, and (i, j) of C at
 * C + i * stride_cm + j * stride_cn (strides in elements) -- the six strides the pages'
 * host wrapper passes its kernel ("Chapter 13: The Blocked Matmul Kernel", section 13.4).
 * A and B strides must be >= 0 (0 repeats a row or column: a broadcast view); C strides
 * must be >= 1 along extents above 1, and no two elements of C may share an address; C may
 * not overlap A or B. A view with a unit stride and a leading stride spanning its lines is
 * read in place (the same path as gemm_run_ex); a column-major C is computed as
 * C^T = B^T A^T in place; any other operand is first gathered into a handle-owned buffer
 * (grown on demand) and any other C is written through a row-major temporary there. Same
 * dtypes, precision modes, errors and stream semantics as gemm_run_ex. */
GEMM_API gemm_status_t gemm_run_strided(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                        const void *A, int64_t stride_am, int64_t stride_ak,
                                        const void *B, int64_t stride_bk, int64_t stride_bn,
                                        void *C, int64_t stride_cm, int64_t stride_cn,
                                        gemm_dtype_t in_dtype, gemm_dtype_t out_dtype,
                                        gemm_precision_t precision_mode, void *cuda_stream);

typedef struct {
  int32_t a_gathered;   /* 1 if A is gathered into the handle's buffer first */
  int32_t b_gathered;   /* 1 if B is gathered */
  int32_t c_mode;       /* 0: C written in place (row-major); 1: C column-major, written in
                           place as C^T = B^T A^T; 2: through a row-major temporary */
  int64_t buffer_bytes; /* handle buffer the call needs for gathers and the temporary */
} gemm_strided_info_t;

/* Host-only: how gemm_run_strided would run these arguments (`info` as gemm_plan fills
 * it for the problem after gathering or transposition; either pointer may be NULL). Same
 * checks and return codes as gemm_run_strided; h may be NULL (default options). */
GEMM_API gemm_status_t gemm_plan_strided(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                         const void *A, int64_t stride_am, int64_t stride_ak,
                                         const void *B, int64_t stride_bk, int64_t stride_bn,
                                         void *C, int64_t stride_cm, int64_t stride_cn,
                                         gemm_dtype_t in_dtype, gemm_dtype_t out_dtype,
                                         gemm_precision_t precision_mode, int32_t sm_count,
                                         gemm_plan_info_t *info, gemm_strided_info_t *sinfo);


/* One piece of a worker's share of the output tiles (see gemm_schedule_segments). */
typedef struct {
  int32_t tile;      /* output tile index in the grouped raster order */
  int32_t kb_begin;  /* first K-block of the tile this piece computes */
  int32_t kb_end;    /* one past its last K-block */
  int32_t role;      /* 0 whole tile, 1 partial (fp32 sum to the workspace), 2 owner (adds
                        the partials of workers first_src..last_src, all numbered below
                        the owner, then stores) */
  int32_t first_src, last_src;
} gemm_segment_t;

/* Host-only view of the tile schedule of the tensor-core kernels: `tiles` output tiles of
 * `k_blocks` K-blocks each on `slots` persistent workers. With stream_k == 0 every tile is
 * done whole, round-robin. Otherwise the tiles of the last, partly filled rounds are cut
 * into K-blocks and shared equally (split-K with a fixed-order reduction: every partial is
 * added by the owner of its tile in increasing worker order). A worker walks its share
 * backwards, so its partial comes first and its owner piece last. Writes worker `slot`'s
 * round-robin tile count to *whole_tiles and up to max_out of its split pieces, in the
 * order the worker computes them, to out; returns the number of split pieces, or -1 for
 * invalid arguments. */
GEMM_API int32_t gemm_schedule_segments(int32_t tiles, int32_t k_blocks, int32_t slots,
                                        int32_t stream_k, int32_t slot, int32_t *whole_tiles,
                                        gemm_segment_t *out, int32_t max_out);

/* Library version as "major.minor.patch". */
GEMM_API const char *gemm_version(void);

/* --------------------------------------------------- allocation-free variant */

/* Size of the fixed device scratch array behind gemm_run_noalloc, in bytes. The first
 * 256 bytes hold a status word; the rest holds staged operand copies. */
#define GEMM_NOALLOC_SCRATCH_BYTES (32u << 20)

/* C = A @ B like gemm_run_ex, for callers that may not allocate device memory at the
 * point of the call -- e.g. a plugin running inside another runtime that owns every
 * device allocation, a deployment that reserves all memory up front and forbids growth,
 * or a host callback / real-time path where cudaMalloc (which can synchronise the
 * device) is not allowed. The pages have no counterpart to this entry point.
 *
 * It takes no handle and allocates nothing: no cudaMalloc, no cudaFree, no allocating
 * library routine. Operands that must be staged (a base or leading dimension TMA cannot
 * address, or an MN-major fp32 operand in tf32 mode) are copied into a file-scope device
 * array of GEMM_NOALLOC_SCRATCH_BYTES that every GPU loading this library keeps until the
 * process exits. Exact fp32 (GEMM_PREC_EXACT_FP32, or DEFAULT with fp32 inputs) also uses
 * that array: beyond the smallest problems (which run on the FMA kernel and need nothing)
 * both operands are split into tf32 hi and lo parts there, about
 * 8 * (M + N) * round_up(K, 32) bytes. A call whose staged copies or split operands would
 * not fit in GEMM_NOALLOC_SCRATCH_BYTES - 256 bytes returns GEMM_ERR_UNSUPPORTED before
 * launching anything (it never falls back to a slower kernel); use gemm_run_ex for it
 * (with GEMM_OPT_FORCE_PATH = 2 for the FMA kernel, which needs no scratch). Arguments
 * and layouts are those of gemm_run_ex; the device is the caller's current device;
 * default options apply, except that tiles are never split along K
 * (GEMM_OPT_STREAM_K = 1: split-K's partial tiles live in a handle's workspace).
 *
 * The first call on each device does a one-time set-up with that device current (it looks
 * up the array's device address and the SM count); make that first call before any
 * stream capture. All calls share the one array and it keeps the last call's contents:
 * two calls that may run at the same time on the GPU (different streams, no ordering
 * between them) race on it. Calls ordered on one stream are safe.
 *
 * device_status: optional caller-owned device int. A device-side bounded wait that
 * expires stores GEMM_ERR_TIMEOUT there (if it still holds 0) and leaves C undefined.
 * With NULL, the status word inside the scratch array is cleared and used instead, and
 * such a failure is not reported. */
GEMM_API gemm_status_t gemm_run_noalloc(int64_t M, int64_t N, int64_t K, const void *A,
                                        int64_t lda, const void *B, int64_t ldb, void *C,
                                        int64_t ldc, gemm_dtype_t in_dtype,
                                        gemm_dtype_t out_dtype, gemm_precision_t precision_mode,
                                        gemm_layout_t a_layout, gemm_layout_t b_layout,
                                        int *device_status, void *cuda_stream);

#ifdef __cplusplus
}
#endif

#endif /* GEMM_GB300_H */
