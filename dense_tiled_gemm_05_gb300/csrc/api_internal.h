// api_internal.h -- what the host runtime's translation units share: the handle, the
// problem and plan types, and the planner / launcher entry points behind include/gemm.h.
// Internal to the library (hidden visibility); not installed.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <vector>

#include "gemm.h"
#include "internal.h"
#include "sk_schedule.h"

// A tuned choice of the tile-shape options for one problem signature (gemm_tune).
struct TuneEntry {
  int64_t M, N, K;
  int in_dtype, out_dtype, precision, a_layout, b_layout;
  gemm_tune_result_t choice;
};

struct gemm_handle_s {
  int device = 0;
  int sm_count = 0;
  int *status = nullptr;  // device status word
  void *workspace = nullptr;
  size_t workspace_bytes = 0;
  uint64_t launches = 0;
  // options
  uint64_t timeout_us = 2000000;
  int force_path = 0;
  int group_m = 8;  // sustained under the power cap, bf16 8192^3: 8 > 16 > 4 > 32
  int max_ctas = 0;
  int stall_producer = 0;
  int force_staging = 0;
  int cta_pair = 0;  // 0 auto, 1 single-CTA tiles, 2 CTA-pair tiles
  int block_n = 0;   // 0 auto, else 128 or 256
  int exact_chunk = 0;  // 0 default
  int acc_chunk = 0;    // fp16-accumulator chunk in K elements, 0 default (16)
  int stage_k = 0;      // 128-byte K-blocks per stage of the CTA-pair kernel, 0 auto
  int tile_rows = 0;    // rows of A per CTA of the CTA-pair kernel, 0 auto
  int stream_k = 0;     // 0 auto (on), 1 off
  int tf32_transpose = 0;  // 1: MN-major tf32 operands staged transposed (K-major)
  int host_panel = 0;  // gemm_run_host panel width (rows of A, columns of B), 0 auto
  // split-K workspace of the CTA-pair kernel: partial tiles and flags
  void *sk_ws = nullptr;
  size_t sk_ws_bytes = 0;
  // host-buffer pipeline (gemm_run_host): device copies of A, B, C, streams and events
  static constexpr int kMaxPanels = 48;  // per operand; steps <= 2 * kMaxPanels
  void *hp_buf = nullptr;
  // six-stride interface (gemm_run_strided): gathered operands and the C temporary
  void *st_buf = nullptr;
  size_t st_bytes = 0;
  size_t hp_bytes = 0;
  cudaStream_t hp_stream[3] = {nullptr, nullptr, nullptr};  // H2D, compute, D2H
  cudaEvent_t hp_event[2 + 4 * kMaxPanels] = {};
  bool hp_ready = false;
  std::vector<TuneEntry> tuned;  // gemm_tune's choices, by problem signature
  // gemm_set_kernel_events: caller's events recorded around the main kernel's launch
  cudaEvent_t kernel_events[2] = {nullptr, nullptr};
};

namespace gemm_gb300 {
namespace api {

// GEMM_LOG=1 prints the failing CUDA call of a GEMM_ERR_CUDA return to stderr.
bool log_enabled();
gemm_status_t cuda_fail(cudaError_t e, const char *what);

// Restores the caller's current device on scope exit.
struct DeviceGuard {
  int prev = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
    if (prev != dev) ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    if (prev >= 0) cudaSetDevice(prev);
  }
};

inline int esize_of(int dt) { return dt == GEMM_F32 ? 4 : 2; }

inline bool valid_dtype(int d) { return d == GEMM_F32 || d == GEMM_F16 || d == GEMM_BF16; }
inline bool valid_layout(int l) { return l == GEMM_ROW_MAJOR || l == GEMM_COL_MAJOR; }

inline int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Byte span [lo, hi) touched by a rows x cols operand with the given layout.
inline void span_of(const void *p, int64_t rows, int64_t cols, int64_t ld, int layout, int es,
             uintptr_t *lo, uintptr_t *hi) {
  const int64_t outer = layout == GEMM_ROW_MAJOR ? rows : cols;
  const int64_t inner = layout == GEMM_ROW_MAJOR ? cols : rows;
  *lo = reinterpret_cast<uintptr_t>(p);
  *hi = *lo + static_cast<uintptr_t>(((outer - 1) * ld + inner) * es);
}

struct Problem {
  int64_t M, N, K;
  const void *A;
  int64_t lda;
  const void *B;
  int64_t ldb;
  void *C;
  int64_t ldc;
  int in_dtype, out_dtype, precision, a_layout, b_layout;
};

struct Options {
  int force_path = 0, group_m = 8, max_ctas = 0, force_staging = 0, cta_pair = 0, block_n = 0;
  int stream_k = 0, exact_chunk = 0, acc_chunk = 0, stage_k = 0, tile_rows = 0;
  int tf32_transpose = 0;
};

// fp16-accumulator chunk (K elements per fp16 rounding of the running total) when the
// caller sets none: the K of one tcgen05.mma.kind::f16.
constexpr int kDefaultAccChunk = 16;

// An operand as the tensor-core kernel sees it: `outer` lines of `inner` contiguous
// elements with leading dimension ld (in elements). It is either read in place or staged
// into the workspace first: copied when TMA cannot address it (misaligned base or
// leading dimension), transposed into K-major form when it is an MN-major operand of a
// kernel that reads K-major operands only (the fp16-accumulator kernel) or a tf32 operand
// under GEMM_OPT_TF32_TRANSPOSE, or split into tf32
// hi/lo parts (exact-fp32 mode; always K-major: [hi | lo], each part K columns
// zero-padded to split_kp, a whole number of 32-long K-blocks).
struct OperandPlan {
  const void *ptr;          // caller's operand
  int64_t ld, outer, inner; // caller's storage: outer lines of inner elements
  bool staged, transpose, split_hl;
  bool is_b, k_contig;      // which operand; whether its storage is K-contiguous
  int64_t rows, k;          // logical rows (M or N) and K, for the split
  int64_t staged_ld;
  int64_t split_kp;         // exact fp32: columns of each part (K rounded up to 32)
  size_t ws_offset, ws_bytes;
  // as read by the kernel (after staging)
  bool mn_major;
  int64_t k_outer, k_inner;
};
struct Plan {
  gemm_plan_info_t info;
  TcVariant variant;
  OperandPlan a, b;
  int fma_tile;
  int chunk_steps;    // chunked tensor-core kernel: MMA instructions per TMEM partial
  int64_t acc_chunk;  // fp16 accumulator: K elements per rounding (0: fp32 accumulator)
  int group_m;        // raster group height (tile rows)
  int stream_k;       // GEMM_OPT_STREAM_K value the plan was made with
  int cta_rows;       // rows of A per CTA (CTA-pair kernel: <= kTcBlockM; else kTcBlockM)
};

struct SplitK {
  gemm_handle_t h = nullptr;
  int mode = 1;  // GEMM_OPT_STREAM_K value
};

// planner.cu
// Flops per byte of A, B and C; under kBandwidthBound the product is bandwidth-bound on
// GB300 (the measured copy bandwidth and bf16 peak put the ridge near 280).
constexpr double kBandwidthBound = 256.0;
double intensity_of(const Problem &P);
gemm_status_t check_args(const Problem &P);
bool use_split_k(int stream_k, int64_t tiles, int64_t k_blocks, int64_t slots);
gemm_status_t make_plan(const Problem &P, const Options &opt, int sm_count, Plan *out);
Options options_of(gemm_handle_t h);
const TuneEntry *find_tuned(gemm_handle_t h, const Problem &P);
Options options_for(gemm_handle_t h, const Problem &P);

// launch.cu
bool encode_2d(CUtensorMap *m, int dtype, const void *base, int64_t inner, int64_t outer,
               int64_t ld, uint32_t box_inner, uint32_t box_outer, bool atom32 = false);
cudaError_t stage_operand(const OperandPlan &o, void *dst, int es, cudaStream_t s);
gemm_status_t launch_tc(const Problem &P, const Plan &pl, const void *a_ptr, int64_t a_ld,
                        const void *b_ptr, int64_t b_ld, int *status, uint64_t timeout_ns,
                        int group_m, int debug_flags, SplitK sk, cudaStream_t s);
// record_events: record the handle's gemm_set_kernel_events pair around the main kernel
// (the calls gemm_set_kernel_events documents; not the host pipeline or the tuner).
gemm_status_t execute(gemm_handle_t h, const Problem &P, const Plan &pl, cudaStream_t s,
                      bool record_events = true);

}  // namespace api
}  // namespace gemm_gb300
