// gemm_api.cu -- host runtime behind include/gemm.h: handle, argument checks, planner,
// operand staging, tensor-map encoding and kernel launch.
//
// The host wrapper of "Chapter 13: The Blocked Matmul Kernel" (section 13.4,
// 01_tiled_matmul.py) reads M, K from A and N from B, checks that the inner dimensions
// agree, lets the caller own C, and launches a (cdiv(M, BLOCK_M), cdiv(N, BLOCK_N)) grid
// with cdiv(K, BLOCK_K) K-iterations per tile. Here the caller states M, N, K and the
// leading dimensions explicitly (the pages pass all six strides), and the planner maps
// the same tile grid onto a persistent schedule of one CTA per SM.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "gemm.h"
#include "internal.h"
#include "sk_schedule.h"

using namespace gemm_gb300;

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
  int group_m = 16;  // gemm_tune chose 16 on bf16 4096^3-8192^3 and tf32 4096^3 (+1-2 %)
  int max_ctas = 0;
  int stall_producer = 0;
  int force_staging = 0;
  int cta_pair = 0;  // 0 auto, 1 single-CTA tiles, 2 CTA-pair tiles
  int block_n = 0;   // 0 auto, else 128 or 256
  int exact_chunk = 0;  // 0 default
  int acc_chunk = 0;    // fp16-accumulator chunk in K elements, 0 default (16)
  int stage_k = 0;      // 128-byte K-blocks per stage of the CTA-pair kernel, 0 auto
  int stream_k = 0;     // 0 auto (on), 1 off
  int host_panel = 0;  // gemm_run_host panel width (rows of A, columns of B), 0 auto
  // split-K workspace of the CTA-pair kernel: partial tiles and flags
  void *sk_ws = nullptr;
  size_t sk_ws_bytes = 0;
  int32_t sk_epoch = 0;
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
};

namespace {

const char *kVersion = "0.1.0";

bool log_enabled() {
  static const bool on = [] {
    const char *e = std::getenv("GEMM_LOG");
    return e && e[0] == '1';
  }();
  return on;
}

gemm_status_t cuda_fail(cudaError_t e, const char *what) {
  if (log_enabled()) std::fprintf(stderr, "[gemm] %s: %s\n", what, cudaGetErrorString(e));
  return GEMM_ERR_CUDA;
}

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

// cuTensorMapEncodeTiled, fetched from the driver through the runtime so the library
// needs no link-time dependency on libcuda.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static std::once_flag once;
  static EncodeTiledFn fn = nullptr;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int esize_of(int dt) { return dt == GEMM_F32 ? 4 : 2; }

bool valid_dtype(int d) { return d == GEMM_F32 || d == GEMM_F16 || d == GEMM_BF16; }
bool valid_layout(int l) { return l == GEMM_ROW_MAJOR || l == GEMM_COL_MAJOR; }

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

// Byte span [lo, hi) touched by a rows x cols operand with the given layout.
void span_of(const void *p, int64_t rows, int64_t cols, int64_t ld, int layout, int es,
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
  int force_path = 0, group_m = 16, max_ctas = 0, force_staging = 0, cta_pair = 0, block_n = 0;
  int stream_k = 0, exact_chunk = 0, acc_chunk = 0, stage_k = 0;
};

// fp16-accumulator chunk (K elements per fp16 rounding of the running total) when the
// caller sets none: the K of one tcgen05.mma.kind::f16.
constexpr int kDefaultAccChunk = 16;

// An operand as the tensor-core kernel sees it: `outer` lines of `inner` contiguous
// elements with leading dimension ld (in elements). It is either read in place or staged
// into the workspace first: copied when TMA cannot address it (misaligned base or
// leading dimension), transposed into K-major form when it is an MN-major operand of a
// kernel that reads K-major operands only (tf32, which the tensor cores take K-major only
// on GB300, and the fp16-accumulator kernel), or split into tf32
// hi/lo parts (exact-fp32 mode; always K-major, 3K columns).
struct OperandPlan {
  const void *ptr;          // caller's operand
  int64_t ld, outer, inner; // caller's storage: outer lines of inner elements
  bool staged, transpose, split3;
  bool is_b, k_contig;      // which operand; whether its storage is K-contiguous
  int64_t rows, k;          // logical rows (M or N) and K, for the split
  int64_t staged_ld;
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
};

gemm_status_t check_args(const Problem &P) {
  if (P.M < 0 || P.N < 0 || P.K < 0) return GEMM_ERR_INVALID_ARG;
  if (!valid_dtype(P.in_dtype) || !valid_dtype(P.out_dtype)) return GEMM_ERR_INVALID_ARG;
  if (!valid_layout(P.a_layout) || !valid_layout(P.b_layout)) return GEMM_ERR_INVALID_ARG;
  if (P.precision < GEMM_PREC_DEFAULT || P.precision > GEMM_PREC_F16_ACC)
    return GEMM_ERR_INVALID_ARG;
  const bool a_used = P.M > 0 && P.K > 0 && P.N > 0;
  const bool b_used = P.K > 0 && P.N > 0 && P.M > 0;
  const bool c_used = P.M > 0 && P.N > 0;
  if (c_used) {
    if (!P.C || P.ldc < P.N) return GEMM_ERR_INVALID_ARG;
  }
  if (a_used) {
    if (!P.A) return GEMM_ERR_INVALID_ARG;
    if (P.lda < (P.a_layout == GEMM_ROW_MAJOR ? P.K : P.M)) return GEMM_ERR_INVALID_ARG;
  }
  if (b_used) {
    if (!P.B) return GEMM_ERR_INVALID_ARG;
    if (P.ldb < (P.b_layout == GEMM_ROW_MAJOR ? P.N : P.K)) return GEMM_ERR_INVALID_ARG;
  }
  if (P.precision == GEMM_PREC_F16_ACC) {
    if (P.in_dtype != GEMM_F16) return GEMM_ERR_UNSUPPORTED;  // the pages' fp16 inputs only
  } else if (P.in_dtype != GEMM_F32 && P.precision != GEMM_PREC_DEFAULT) {
    return GEMM_ERR_UNSUPPORTED;
  }
  if (P.M > INT32_MAX || P.N > INT32_MAX || P.K > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
  const int es = esize_of(P.in_dtype), os = esize_of(P.out_dtype);
  if ((a_used && reinterpret_cast<uintptr_t>(P.A) % es) ||
      (b_used && reinterpret_cast<uintptr_t>(P.B) % es) ||
      (c_used && reinterpret_cast<uintptr_t>(P.C) % os))
    return GEMM_ERR_ALIGNMENT;
  if (c_used) {
    uintptr_t clo, chi;
    span_of(P.C, P.M, P.N, P.ldc, GEMM_ROW_MAJOR, os, &clo, &chi);
    if (a_used) {
      uintptr_t lo, hi;
      span_of(P.A, P.M, P.K, P.lda, P.a_layout, es, &lo, &hi);
      if (clo < hi && lo < chi) return GEMM_ERR_INVALID_ARG;
    }
    if (b_used) {
      uintptr_t lo, hi;
      span_of(P.B, P.K, P.N, P.ldb, P.b_layout, es, &lo, &hi);
      if (clo < hi && lo < chi) return GEMM_ERR_INVALID_ARG;
    }
  }
  return GEMM_OK;
}

// TMA can read an operand in place when its base is 16-byte aligned and its leading
// dimension is a multiple of 16 bytes (a single line needs no stride).
bool tma_legal(const void *p, int64_t ld, int64_t outer, int es) {
  if (reinterpret_cast<uintptr_t>(p) % 16) return false;
  return outer <= 1 || (ld * es) % 16 == 0;
}

OperandPlan plan_operand(const void *p, int64_t rows, int64_t cols, int64_t ld, int layout,
                         bool k_is_rows_dim, int es, bool force_stage, bool split3,
                         bool k_major_only, size_t *ws_cursor) {
  OperandPlan o{};
  o.ptr = p;
  o.ld = ld;
  o.outer = layout == GEMM_ROW_MAJOR ? rows : cols;
  o.inner = layout == GEMM_ROW_MAJOR ? cols : rows;
  // The operand is K-major when K is its contiguous axis.
  const bool k_inner = k_is_rows_dim ? layout == GEMM_COL_MAJOR : layout == GEMM_ROW_MAJOR;
  o.is_b = k_is_rows_dim;
  o.k_contig = k_inner;
  o.rows = k_is_rows_dim ? cols : rows;
  o.k = k_is_rows_dim ? rows : cols;
  o.mn_major = !k_inner;
  o.k_outer = o.outer;
  o.k_inner = o.inner;
  o.split3 = split3;
  o.transpose = !split3 && o.mn_major && (es == 4 || k_major_only);
  o.staged = split3 || o.transpose || force_stage || !tma_legal(p, ld, o.outer, es);
  if (o.staged) {
    if (split3) {
      o.k_outer = o.rows;
      o.k_inner = 3 * o.k;
      o.mn_major = false;
    } else if (o.transpose) {
      o.k_outer = o.inner;
      o.k_inner = o.outer;
      o.mn_major = false;
    }
    o.staged_ld = round_up(o.k_inner, 16 / es);
    o.ws_offset = *ws_cursor;
    o.ws_bytes = static_cast<size_t>(o.staged_ld * o.k_outer * es);
    *ws_cursor = static_cast<size_t>(round_up(static_cast<int64_t>(*ws_cursor + o.ws_bytes), 256));
  }
  return o;
}

// Whether splitting the last rounds along K pays on GB300 (interleaved measurements of
// bf16 products): it does when at least two whole rounds come first and every tile has a
// long K-loop (4096^3 +5.6 %, 5120^3 +7.4 %, 8192^3 +3.6 %); it does not when every tile
// has to be split (2048^3 -26 %) or K is short (8192 x 8192 x 2048 -1.6 %), where the
// partial-tile traffic costs more than the idle tail it saves. stream_k: 0 by this rule,
// 1 never, 2 whenever the schedule allows.
bool use_split_k(int stream_k, int64_t tiles, int64_t k_blocks, int64_t slots) {
  if (stream_k == 1) return false;
  if (stream_k == 2) return true;
  return slots > 0 && tiles % slots != 0 && tiles / slots >= 2 && k_blocks >= 64;
}

// Tile width by a wave-quantisation cost model: a persistent grid runs
// ceil(tiles / slots) rounds, each as long as one tile. A 128-wide tile has half the
// flops of a 256-wide one but, measured on GB300, takes about 0.75 of its time (every MMA
// re-reads its 128 x 16 slice of A from shared memory, so narrow MMAs are starved of
// shared-memory bandwidth); it wins only when it fills the machine much better, e.g.
// when N itself is at most 128.
int pick_block_n(int64_t M, int64_t N, int64_t k_blocks, bool pair, int stream_k, int sm_count) {
  const int64_t rows = pair ? 2 * kTcBlockM : kTcBlockM;
  const int64_t slots = pair ? (sm_count > 1 ? sm_count / 2 : 1) : (sm_count > 0 ? sm_count : 1);
  const int64_t tiles_m = (M + rows - 1) / rows;
  auto cost = [&](int64_t bn, double per_column) {
    const int64_t tiles = tiles_m * ((N + bn - 1) / bn);
    // With a split-K share the last round is spread over every slot: fractional rounds.
    const bool split = pair && use_split_k(stream_k, tiles, k_blocks, slots) &&
                       sk_dp_tiles(static_cast<int32_t>(tiles), static_cast<int32_t>(k_blocks),
                                   static_cast<int32_t>(slots), true) < tiles;
    const double rounds = split ? static_cast<double>(tiles) / static_cast<double>(slots)
                                : static_cast<double>((tiles + slots - 1) / slots);
    return rounds * static_cast<double>(bn) * per_column;
  };
  return cost(128, 1.5) < cost(256, 1.0) ? 128 : 256;
}

gemm_status_t make_plan(const Problem &P, const Options &opt, int sm_count, Plan *out) {
  gemm_status_t st = check_args(P);
  if (st != GEMM_OK) return st;
  Plan pl{};
  pl.group_m = opt.group_m;
  pl.stream_k = opt.stream_k;
  gemm_plan_info_t &I = pl.info;
  if (P.M == 0 || P.N == 0) {
    I.path = GEMM_PATH_NONE;
    *out = pl;
    return GEMM_OK;
  }
  if (P.K == 0) {
    I.path = GEMM_PATH_ZERO_FILL;
    I.ctas = 1;
    *out = pl;
    return GEMM_OK;
  }
  // Exact fp32 runs on the tensor cores as three tf32 products of split operands, except
  // for tiny problems (the pages' 8 x 8 example and smaller), which take the fp32 FMA
  // kernel with 4 x 4 x 4 tiles; GEMM_OPT_FORCE_PATH chooses either explicitly. The fp16
  // accumulator runs on the tensor cores when its chunk is a whole number of 16-long MMAs,
  // else (e.g. the pages' BLOCK_K = 8) on the FMA kernel, whose K-tile is 8.
  const bool exact = P.in_dtype == GEMM_F32 && P.precision != GEMM_PREC_TF32;
  const bool f16acc = P.precision == GEMM_PREC_F16_ACC;
  pl.acc_chunk = f16acc ? (opt.acc_chunk > 0 ? opt.acc_chunk : kDefaultAccChunk) : 0;
  bool use_fma = (exact && P.M * P.N <= 256) || (f16acc && pl.acc_chunk % 16 != 0);
  if (opt.force_path == 2) use_fma = true;
  if (opt.force_path == 1) {
    if (f16acc && pl.acc_chunk % 16 != 0) return GEMM_ERR_UNSUPPORTED;
    use_fma = false;
  }
  const bool split = exact && !use_fma;
  if (use_fma) {
    pl.fma_tile = (P.M * P.N <= 256 && !f16acc) ? 4 : 128;
    int bm, bn, bk;
    fma_tile_shape(pl.fma_tile, &bm, &bn, &bk);
    if (pl.acc_chunk % bk) return GEMM_ERR_UNSUPPORTED;
    I.path = GEMM_PATH_FMA;
    I.tile_m = bm, I.tile_n = bn, I.tile_k = bk;
    I.grid_m = (P.M + bm - 1) / bm;
    I.grid_n = (P.N + bn - 1) / bn;
    I.k_iters = (P.K + bk - 1) / bk;
    if (I.grid_m > 65535 || I.grid_n > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    I.ctas = I.grid_m * I.grid_n;
    *out = pl;
    return GEMM_OK;
  }
  const int es = esize_of(P.in_dtype);
  const int os = esize_of(P.out_dtype);
  size_t cursor = 0;
  pl.a = plan_operand(P.A, P.M, P.K, P.lda, P.a_layout, false, es, opt.force_staging != 0, split,
                      f16acc, &cursor);
  pl.b = plan_operand(P.B, P.K, P.N, P.ldb, P.b_layout, true, es, opt.force_staging != 0, split,
                      f16acc, &cursor);
  pl.variant.esize = es;
  pl.variant.a_mn = pl.a.mn_major;
  pl.variant.b_mn = pl.b.mn_major;
  // Flops per byte of A, B and C: under ~256 the product is bandwidth-bound on GB300.
  const double intensity = 2.0 * P.M * P.N * P.K /
                           (es * (static_cast<double>(P.M) * P.K + static_cast<double>(P.K) * P.N) +
                            static_cast<double>(os) * P.M * P.N);
  // CTA pairs (256-row tiles on two SMs) halve the shared-memory and L2 traffic per
  // flop; a problem no taller than one 128-row tile keeps single-CTA tiles, and so does a
  // compute-bound one whose 128 x 256 single-CTA tiles all run at once (one round on the
  // SMs), where the pair's cross-SM handshakes cost more than they save (bf16 2048^3:
  // 16.6 against 18.7 us). Bandwidth-bound ones keep pairs, for their wide stages.
  const int64_t single_tiles = ((P.M + kTcBlockM - 1) / kTcBlockM) * ((P.N + 255) / 256);
  const bool one_round = single_tiles <= sm_count && intensity >= 256.0;
  pl.variant.pair = opt.cta_pair == 2 || (opt.cta_pair == 0 && P.M > kTcBlockM && !one_round);
  pl.variant.block_n =
      opt.block_n ? opt.block_n
                  : pick_block_n(P.M, P.N, (P.K + 128 / es - 1) / (128 / es), pl.variant.pair,
                                 split ? 1 : opt.stream_k, sm_count);
  if (split || f16acc) {  // the chunked kernel has one shape: CTA pairs, 256 x 256 tiles
    pl.variant.exact = split;
    pl.variant.f16acc = f16acc;
    pl.variant.pair = true;
    pl.variant.block_n = 256;
  }
  const bool chunked = pl.variant.exact || pl.variant.f16acc;
  // Two 128-byte K-blocks per stage (CTA-pair kernel, K-major 16-bit operands): each row
  // of A and B is then fetched 256 contiguous bytes at a time. By default only for
  // bandwidth-bound products (under ~256 flops per byte of A, B and C), where it measured
  // +1.5 % on bf16 16384 x 128 x 8192; compute-bound ones keep the deeper ring of one
  // K-block per stage (4096^3 lost 9 % with wide stages). A forced split-K keeps narrow
  // K-blocks, the finer unit it shares out (one 256 x 256 x 8192 tile: 128 units for 76
  // clusters rather than 64).
  const bool wide_ok = pl.variant.pair && !chunked && es == 2 && !pl.a.mn_major && !pl.b.mn_major;
  if (opt.stage_k == 2 && !wide_ok) return GEMM_ERR_UNSUPPORTED;
  pl.variant.kps =
      opt.stage_k == 2 || (opt.stage_k == 0 && wide_ok && intensity < 256.0 && opt.stream_k != 2)
          ? 2
          : 1;
  I.path = split ? GEMM_PATH_TCGEN05_3XTF32 : f16acc ? GEMM_PATH_TCGEN05_F16ACC : GEMM_PATH_TCGEN05;
  I.tile_m = pl.variant.pair ? 2 * kTcBlockM : kTcBlockM;
  I.tile_n = pl.variant.block_n;
  I.tile_k = pl.variant.kps * 128 / es;
  I.grid_m = (P.M + I.tile_m - 1) / I.tile_m;
  I.grid_n = (P.N + I.tile_n - 1) / I.tile_n;
  const int64_t k_total = split ? 3 * P.K : P.K;  // split operands concatenate 3 products
  I.k_iters = (k_total + I.tile_k - 1) / I.tile_k;
  if (I.grid_m * I.grid_n > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
  // chunked kernel: four MMAs per 128-byte K-block
  if (split)
    pl.chunk_steps = 4 * (opt.exact_chunk > 0 ? opt.exact_chunk : exact_chunk_kblocks(I.k_iters));
  else if (f16acc)
    pl.chunk_steps = static_cast<int>(pl.acc_chunk / 16);
  I.stages = tc_stages(pl.variant);
  I.stage_a = pl.a.staged, I.stage_b = pl.b.staged;
  I.a_mn_major = pl.a.mn_major, I.b_mn_major = pl.b.mn_major;
  // TMA stores need a 16-byte aligned base and row pitch; they are also used only when a
  // row of C ends on a 16-byte boundary, because a store box clipped at a right edge that
  // falls inside a 16-byte granule was seen to write the whole granule (past column N).
  I.tma_store = reinterpret_cast<uintptr_t>(P.C) % 16 == 0 && (P.ldc * os) % 16 == 0 &&
                (P.N * os) % 16 == 0;
  const int64_t tiles = I.grid_m * I.grid_n;
  if (pl.variant.pair) {
    // One cluster of two CTAs per tile slot; the launch clamps to the clusters that fit.
    // With a split-K share every cluster takes part, even when there are fewer tiles.
    int64_t clusters = sm_count > 1 ? sm_count / 2 : 1;
    if (opt.max_ctas > 0 && opt.max_ctas / 2 < clusters) clusters = opt.max_ctas / 2 > 0 ? opt.max_ctas / 2 : 1;
    // (the fp16 accumulator never splits: its running total takes the chunks in order)
    const bool split = !pl.variant.f16acc && use_split_k(opt.stream_k, tiles, I.k_iters, clusters) &&
                       sk_dp_tiles(static_cast<int32_t>(tiles), static_cast<int32_t>(I.k_iters),
                                   static_cast<int32_t>(clusters), true) < tiles;
    I.ctas = 2 * (split || tiles > clusters ? clusters : tiles);
  } else {
    int64_t ctas = sm_count > 0 ? sm_count : 1;
    if (opt.max_ctas > 0 && opt.max_ctas < ctas) ctas = opt.max_ctas;
    I.ctas = tiles < ctas ? tiles : ctas;
  }
  I.workspace_bytes = static_cast<int64_t>(cursor);
  I.cta_pair = pl.variant.pair ? 1 : 0;
  if (pl.variant.pair && !pl.variant.f16acc) {
    const int32_t slots = static_cast<int32_t>(I.ctas / 2);
    const int32_t t = static_cast<int32_t>(tiles);
    if (use_split_k(opt.stream_k, t, I.k_iters, slots))
      I.split_tiles = t - sk_dp_tiles(t, static_cast<int32_t>(I.k_iters), slots, true);
  }
  *out = pl;
  return GEMM_OK;
}

CUtensorMapDataType tmap_dtype(int dt) {
  switch (dt) {
    case GEMM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case GEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  }
}

// 2D tensor map: dims {inner, outer}, row pitch ld elements, box {box_inner, box_outer},
// 128-byte swizzle, zero fill outside the tensor.
bool encode_2d(CUtensorMap *m, int dtype, const void *base, int64_t inner, int64_t outer,
               int64_t ld, uint32_t box_inner, uint32_t box_outer) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const int es = esize_of(dtype);
  int64_t pitch = ld * es;
  if (outer <= 1) pitch = round_up(inner * es, 16);  // a single line: any legal pitch
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch)};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, tmap_dtype(dtype), 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS && log_enabled())
    std::fprintf(stderr, "[gemm] cuTensorMapEncodeTiled failed (%d)\n", static_cast<int>(r));
  return r == CUDA_SUCCESS;
}

uint32_t make_idesc(int in_dtype, bool a_mn, bool b_mn, int n, int m) {
  const uint32_t fmt = in_dtype == GEMM_F16 ? 0u : in_dtype == GEMM_BF16 ? 1u : 2u;
  uint32_t d = 0;
  d |= 1u << 4;                               // accumulator: f32
  d |= fmt << 7;                              // A format
  d |= fmt << 10;                             // B format
  d |= (a_mn ? 1u : 0u) << 15;                // A major-ness (1 = MN-major)
  d |= (b_mn ? 1u : 0u) << 16;                // B major-ness
  d |= static_cast<uint32_t>(n >> 3) << 17;   // N / 8
  d |= static_cast<uint32_t>(m >> 4) << 24;   // M / 16
  return d;
}

gemm_status_t ensure_workspace(gemm_handle_t h, size_t bytes) {
  if (bytes <= h->workspace_bytes) return GEMM_OK;
  const char *fi = std::getenv("GEMM_FAULT_INJECT");
  if (fi && std::strcmp(fi, "alloc") == 0) return GEMM_ERR_NO_MEMORY;
  if (h->workspace) {
    cudaFree(h->workspace);  // synchronises: no launched work still uses it
    h->workspace = nullptr;
    h->workspace_bytes = 0;
  }
  void *p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_MEMORY;
  }
  h->workspace = p;
  h->workspace_bytes = bytes;
  return GEMM_OK;
}

Options options_of(gemm_handle_t h) {
  Options o;
  if (h) {
    o.force_path = h->force_path;
    o.group_m = h->group_m;
    o.max_ctas = h->max_ctas;
    o.force_staging = h->force_staging;
    o.cta_pair = h->cta_pair;
    o.block_n = h->block_n;
    o.stream_k = h->stream_k;
    o.exact_chunk = h->exact_chunk;
    o.acc_chunk = h->acc_chunk;
    o.stage_k = h->stage_k;
  }
  return o;
}

const TuneEntry *find_tuned(gemm_handle_t h, const Problem &P) {
  if (!h) return nullptr;
  for (const TuneEntry &t : h->tuned)
    if (t.M == P.M && t.N == P.N && t.K == P.K && t.in_dtype == P.in_dtype &&
        t.out_dtype == P.out_dtype && t.precision == P.precision && t.a_layout == P.a_layout &&
        t.b_layout == P.b_layout)
      return &t;
  return nullptr;
}

// The handle's options, with the tile-shape options gemm_tune chose for this problem
// signature (if it was tuned) in place of the handle's.
Options options_for(gemm_handle_t h, const Problem &P) {
  Options o = options_of(h);
  if (const TuneEntry *t = find_tuned(h, P)) {
    o.cta_pair = t->choice.cta_pair;
    o.block_n = t->choice.block_n;
    o.stream_k = t->choice.stream_k;
    o.stage_k = t->choice.stage_k;
    o.group_m = t->choice.group_m;
  }
  return o;
}

cudaError_t stage_operand(const OperandPlan &o, void *dst, int es, cudaStream_t s) {
  if (o.split3)
    return split3_launch(static_cast<const float *>(o.ptr), o.ld, o.k_contig,
                         static_cast<float *>(dst), o.staged_ld, o.rows, o.k, o.is_b, s);
  if (o.transpose) return transpose_launch(o.ptr, o.ld, dst, o.staged_ld, o.outer, o.inner, es, s);
  return repack_launch(o.ptr, o.ld, dst, o.staged_ld, o.outer, o.inner, es, s);
}

// Tensor maps, kernel parameters and launch of the tensor-core kernel for operands that
// are already TMA-legal (in place or staged).
// Split-K context of a launch: a workspace provider (null = split-K off).
struct SplitK {
  gemm_handle_t h = nullptr;
  int mode = 1;  // GEMM_OPT_STREAM_K value
};

gemm_status_t ensure_sk_workspace(gemm_handle_t h, size_t bytes, size_t flag_bytes,
                                  cudaStream_t s) {
  if (bytes <= h->sk_ws_bytes) return GEMM_OK;
  if (h->sk_ws) {
    cudaFree(h->sk_ws);
    h->sk_ws = nullptr;
    h->sk_ws_bytes = 0;
  }
  void *p = nullptr;
  if (cudaMalloc(&p, bytes) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_NO_MEMORY;
  }
  // Flags start at 0 and every launch uses a fresh non-zero epoch, so stale flags of
  // earlier launches never match.
  if (cudaMemsetAsync(p, 0, flag_bytes, s) != cudaSuccess) {
    cudaFree(p);
    return GEMM_ERR_CUDA;
  }
  h->sk_ws = p;
  h->sk_ws_bytes = bytes;
  return GEMM_OK;
}

gemm_status_t launch_tc(const Problem &P, const Plan &pl, const void *a_ptr, int64_t a_ld,
                        const void *b_ptr, int64_t b_ld, int *status, uint64_t timeout_ns,
                        int group_m, int debug_flags, SplitK sk, cudaStream_t s) {
  const gemm_plan_info_t &I = pl.info;
  const int es = esize_of(P.in_dtype);
  const uint32_t row_elems = 128 / es;  // elements in one 128-byte swizzle row
  CUtensorMap tmA, tmB, tmC, tmP;
  std::memset(&tmC, 0, sizeof tmC);
  std::memset(&tmP, 0, sizeof tmP);
  // K-major operand: box = (one 128-byte row of K) x (the CTA's rows of the tile);
  // MN-major operand: box = (one 128-byte row of M or N) x (the stage's K rows).
  const uint32_t cta_rows_a = kTcBlockM;
  const uint32_t cta_rows_b = pl.variant.pair ? I.tile_n / 2 : I.tile_n;
  const uint32_t a_box_outer = pl.a.mn_major ? row_elems : cta_rows_a;
  const uint32_t b_box_outer = pl.b.mn_major ? row_elems : cta_rows_b;
  if (!encode_2d(&tmA, P.in_dtype, a_ptr, pl.a.k_inner, pl.a.k_outer, a_ld, row_elems,
                 a_box_outer) ||
      !encode_2d(&tmB, P.in_dtype, b_ptr, pl.b.k_inner, pl.b.k_outer, b_ld, row_elems,
                 b_box_outer))
    return GEMM_ERR_CUDA;
  if (I.tma_store) {
    const uint32_t out_row = 128 / esize_of(P.out_dtype);
    if (!encode_2d(&tmC, P.out_dtype, P.C, P.N, P.M, P.ldc, out_row, 32)) return GEMM_ERR_CUDA;
  }
  TcParams tp{};
  tp.M = static_cast<int32_t>(P.M);
  tp.N = static_cast<int32_t>(P.N);
  tp.K = static_cast<int32_t>(P.K);
  tp.tiles_m = static_cast<int32_t>(I.grid_m);
  tp.tiles_n = static_cast<int32_t>(I.grid_n);
  tp.k_blocks = static_cast<int32_t>(I.k_iters);
  tp.group_m = static_cast<int32_t>(group_m < I.grid_m ? group_m : I.grid_m);
  tp.idesc = make_idesc(P.in_dtype, pl.a.mn_major, pl.b.mn_major, I.tile_n, I.tile_m);
  tp.out_dtype = P.out_dtype;
  tp.tma_store = I.tma_store;
  tp.C = P.C;
  tp.ldc = P.ldc;
  tp.status = status;
  tp.timeout_ns = timeout_ns;
  tp.debug_flags = debug_flags;
  tp.chunk_steps = pl.chunk_steps;
  int64_t grid = I.ctas;
  if (pl.variant.pair) {
    const int64_t fit = pl.variant.exact || pl.variant.f16acc
                            ? tc_chunk_max_active_clusters(pl.variant.f16acc)
                            : tc2_max_active_clusters();
    if (fit <= 0) return GEMM_ERR_CUDA;
    if (grid / 2 > fit) grid = 2 * fit;
  }
  // Split-K share of the last rounds (CTA-pair kernel): whole tiles otherwise.
  const int32_t tiles = tp.tiles_m * tp.tiles_n;
  tp.sk_dp_tiles = tiles;
  if (pl.variant.pair && !pl.variant.f16acc && sk.h) {
    const int32_t slots = static_cast<int32_t>(grid / 2);
    tp.sk_dp_tiles = sk_dp_tiles(tiles, tp.k_blocks, slots,
                                 use_split_k(sk.mode, tiles, tp.k_blocks, slots));
    if (tp.sk_dp_tiles < tiles) {
      // one flag per epilogue warp of each CTA (4 in the CTA-pair kernel, 8 in the chunked one)
      const size_t flag_bytes = static_cast<size_t>(slots) * 2 * 8 * sizeof(int);
      const size_t flag_region = (flag_bytes + 255) / 256 * 256;
      const size_t part_bytes =
          static_cast<size_t>(slots) * 2 * kTcBlockM * pl.variant.block_n * sizeof(float);
      gemm_status_t st = ensure_sk_workspace(sk.h, flag_region + part_bytes, flag_region, s);
      if (st != GEMM_OK) return st;
      tp.sk_flags = static_cast<int *>(sk.h->sk_ws);
      tp.sk_partials = reinterpret_cast<float *>(static_cast<char *>(sk.h->sk_ws) + flag_region);
      // partial tiles: rows [worker][cta rank][128], block_n fp32 columns; 32 x 32 boxes
      if (!encode_2d(&tmP, GEMM_F32, tp.sk_partials, pl.variant.block_n,
                     static_cast<int64_t>(slots) * 2 * kTcBlockM, pl.variant.block_n, 32, 32))
        return GEMM_ERR_CUDA;
      sk.h->sk_epoch = sk.h->sk_epoch == INT32_MAX ? 1 : sk.h->sk_epoch + 1;
      tp.sk_epoch = sk.h->sk_epoch;
    }
  }
  const cudaError_t e = tc_launch(pl.variant, tmA, tmB, tmC, tmP, tp, static_cast<int>(grid), s);
  return e == cudaSuccess ? GEMM_OK : cuda_fail(e, "tcgen05 launch");
}

gemm_status_t execute(gemm_handle_t h, const Problem &P, const Plan &pl, cudaStream_t s) {
  const gemm_plan_info_t &I = pl.info;
  cudaError_t e;
  switch (I.path) {
    case GEMM_PATH_NONE: return GEMM_OK;
    case GEMM_PATH_ZERO_FILL:
      e = zero_fill_launch(P.C, P.ldc, P.M, P.N, P.out_dtype, s);
      if (e != cudaSuccess) return cuda_fail(e, "zero fill launch");
      h->launches += 1;
      return GEMM_OK;
    case GEMM_PATH_FMA: {
      FmaParams fp{P.M, P.N, P.K, P.A, P.lda, P.B, P.ldb, P.C, P.ldc, P.in_dtype, P.out_dtype,
                   P.a_layout == GEMM_COL_MAJOR, P.b_layout == GEMM_COL_MAJOR, pl.acc_chunk};
      e = fma_launch(fp, pl.fma_tile, s);
      if (e != cudaSuccess) return cuda_fail(e, "fma launch");
      h->launches += 1;
      return GEMM_OK;
    }
    default: break;
  }
  // Tensor-core path.
  const int es = esize_of(P.in_dtype);
  gemm_status_t st = ensure_workspace(h, static_cast<size_t>(I.workspace_bytes));
  if (st != GEMM_OK) return st;
  const void *a_ptr = pl.a.ptr;
  int64_t a_ld = pl.a.ld;
  const void *b_ptr = pl.b.ptr;
  int64_t b_ld = pl.b.ld;
  for (const OperandPlan *o : {&pl.a, &pl.b}) {
    if (!o->staged) continue;
    void *dst = static_cast<char *>(h->workspace) + o->ws_offset;
    e = stage_operand(*o, dst, es, s);
    if (e != cudaSuccess) return cuda_fail(e, "stage operand");
    h->launches += 1;
    if (o == &pl.a)
      a_ptr = dst, a_ld = o->staged_ld;
    else
      b_ptr = dst, b_ld = o->staged_ld;
  }
  SplitK sk;
  sk.h = h;
  sk.mode = pl.stream_k;
  st = launch_tc(P, pl, a_ptr, a_ld, b_ptr, b_ld, h->status, h->timeout_us * 1000ull,
                 pl.group_m, h->stall_producer ? kDebugStallProducer : 0, sk, s);
  if (st != GEMM_OK) return st;
  h->launches += 1;
  return GEMM_OK;
}

}  // namespace

extern "C" {

GEMM_API const char *gemm_version(void) { return kVersion; }

GEMM_API int32_t gemm_schedule_segments(int32_t tiles, int32_t k_blocks, int32_t slots,
                                        int32_t stream_k, int32_t slot, int32_t *whole_tiles,
                                        gemm_segment_t *out, int32_t max_out) {
  if (tiles < 0 || k_blocks < 1 || slots < 1 || slot < 0 || slot >= slots || max_out < 0)
    return -1;
  const SkSchedule S =
      sk_make(tiles, k_blocks, slots, sk_dp_tiles(tiles, k_blocks, slots, stream_k != 0));
  if (whole_tiles) *whole_tiles = sk_dp_count(S, slot);
  int32_t n = 0;
  for (int64_t lo = sk_begin(S, slot), hi = sk_begin(S, slot + 1); hi > lo; ++n) {
    SkSegment seg;
    hi = sk_segment_at(S, slot, hi, &seg);
    if (out && n < max_out)
      out[n] = gemm_segment_t{seg.tile, seg.kb_begin, seg.kb_end, seg.role, seg.first_src,
                              seg.last_src};
  }
  return n;
}

GEMM_API const char *gemm_strerror(gemm_status_t s) {
  switch (s) {
    case GEMM_OK: return "success";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_UNSUPPORTED: return "unsupported request";
    case GEMM_ERR_ALIGNMENT: return "pointer not aligned to its element size";
    case GEMM_ERR_NO_MEMORY: return "workspace allocation failed";
    case GEMM_ERR_CUDA: return "CUDA call failed";
    case GEMM_ERR_TIMEOUT: return "device-side bounded wait expired";
    case GEMM_ERR_DEVICE: return "no usable sm_103 device";
  }
  return "unknown status";
}

GEMM_API gemm_status_t gemm_create(gemm_handle_t *out, int device) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  int n = 0;
  if (cudaGetDeviceCount(&n) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_DEVICE;
  }
  if (device < 0 || device >= n) return GEMM_ERR_DEVICE;
  cudaDeviceProp prop;
  if (cudaGetDeviceProperties(&prop, device) != cudaSuccess) return GEMM_ERR_CUDA;
  if (prop.major != 10 || prop.minor != 3) return GEMM_ERR_DEVICE;  // built for sm_103a only
  DeviceGuard g(device);
  if (!g.ok) return GEMM_ERR_CUDA;
  gemm_handle_t h = new (std::nothrow) gemm_handle_s();
  if (!h) return GEMM_ERR_NO_MEMORY;
  h->device = device;
  h->sm_count = prop.multiProcessorCount;
  if (cudaMalloc(&h->status, sizeof(int)) != cudaSuccess ||
      cudaMemset(h->status, 0, sizeof(int)) != cudaSuccess) {
    cudaGetLastError();
    if (h->status) cudaFree(h->status);
    delete h;
    return GEMM_ERR_NO_MEMORY;
  }
  *out = h;
  return GEMM_OK;
}

GEMM_API void gemm_destroy(gemm_handle_t h) {
  if (!h) return;
  DeviceGuard g(h->device);
  cudaDeviceSynchronize();
  if (h->workspace) cudaFree(h->workspace);
  if (h->sk_ws) cudaFree(h->sk_ws);
  if (h->hp_buf) cudaFree(h->hp_buf);
  if (h->st_buf) cudaFree(h->st_buf);
  if (h->hp_ready) {
    for (cudaStream_t st : h->hp_stream) cudaStreamDestroy(st);
    for (cudaEvent_t ev : h->hp_event) cudaEventDestroy(ev);
  }
  if (h->status) cudaFree(h->status);
  delete h;
}

GEMM_API gemm_status_t gemm_set_option(gemm_handle_t h, gemm_option_t opt, int64_t v) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  switch (opt) {
    case GEMM_OPT_WAIT_TIMEOUT_US:
      if (v < 1 || v > 600000000) return GEMM_ERR_INVALID_ARG;
      h->timeout_us = static_cast<uint64_t>(v);
      return GEMM_OK;
    case GEMM_OPT_FORCE_PATH:
      if (v < 0 || v > 2) return GEMM_ERR_INVALID_ARG;
      h->force_path = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_GROUP_M:
      if (v < 1 || v > 65536) return GEMM_ERR_INVALID_ARG;
      h->group_m = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_MAX_CTAS:
      if (v < 0 || v > 1 << 20) return GEMM_ERR_INVALID_ARG;
      h->max_ctas = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_FAULT_STALL_PRODUCER:
      if (v < 0 || v > 1) return GEMM_ERR_INVALID_ARG;
      h->stall_producer = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_FORCE_STAGING:
      if (v < 0 || v > 1) return GEMM_ERR_INVALID_ARG;
      h->force_staging = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_CTA_PAIR:
      if (v < 0 || v > 2) return GEMM_ERR_INVALID_ARG;
      h->cta_pair = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_STAGE_K:
      if (v < 0 || v > 2) return GEMM_ERR_INVALID_ARG;
      h->stage_k = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_ACC_CHUNK:
      if (v < 0 || v > (int64_t{1} << 20) || v % 8) return GEMM_ERR_INVALID_ARG;
      h->acc_chunk = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_HOST_PANEL:
      if (v < 0 || v > (int64_t{1} << 30) || v % 256) return GEMM_ERR_INVALID_ARG;
      h->host_panel = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_STREAM_K:
      if (v < 0 || v > 2) return GEMM_ERR_INVALID_ARG;
      h->stream_k = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_EXACT_CHUNK:
      if (v < 0 || v > 64) return GEMM_ERR_INVALID_ARG;
      h->exact_chunk = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_BLOCK_N:
      if (v != 0 && v != 128 && v != 256) return GEMM_ERR_INVALID_ARG;
      h->block_n = static_cast<int>(v);
      return GEMM_OK;
  }
  return GEMM_ERR_INVALID_ARG;
}

GEMM_API gemm_status_t gemm_get_launch_count(gemm_handle_t h, uint64_t *count) {
  if (!h || !count) return GEMM_ERR_INVALID_ARG;
  *count = h->launches;
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_plan(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void *A,
                                 int64_t lda, const void *B, int64_t ldb, void *C, int64_t ldc,
                                 gemm_dtype_t in_dtype, gemm_dtype_t out_dtype,
                                 gemm_precision_t precision_mode, gemm_layout_t a_layout,
                                 gemm_layout_t b_layout, int32_t sm_count, gemm_plan_info_t *info) {
  if (!info) return GEMM_ERR_INVALID_ARG;
  const Problem P{M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, precision_mode, a_layout,
                  b_layout};
  Plan pl;
  gemm_status_t st = make_plan(P, options_for(h, P), sm_count, &pl);
  if (st == GEMM_OK) *info = pl.info;
  return st;
}

GEMM_API gemm_status_t gemm_run_ex(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                   const void *A, int64_t lda, const void *B, int64_t ldb,
                                   void *C, int64_t ldc, gemm_dtype_t in_dtype,
                                   gemm_dtype_t out_dtype, gemm_precision_t precision_mode,
                                   gemm_layout_t a_layout, gemm_layout_t b_layout,
                                   void *cuda_stream) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  const Problem P{M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, precision_mode, a_layout,
                  b_layout};
  Plan pl;
  gemm_status_t st = make_plan(P, options_for(h, P), h->sm_count, &pl);
  if (st != GEMM_OK) return st;
  DeviceGuard g(h->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  return execute(h, P, pl, static_cast<cudaStream_t>(cuda_stream));
}

// ------------------------------------------------------------------ tuning
//
// The pages choose BLOCK_M/N/K per call; here the planner picks the tile shape, the
// split-K share, the stage width and the raster group by fixed rules. gemm_tune measures
// the alternatives for one problem on the device and keeps the fastest for its signature.

namespace {

gemm_tune_result_t choice_of(const Options &o, const Plan &pl) {
  gemm_tune_result_t c{};
  c.cta_pair = pl.variant.pair ? 2 : 1;
  c.block_n = pl.variant.block_n;
  c.stream_k = o.stream_k;
  c.stage_k = pl.variant.kps;
  c.group_m = o.group_m;
  return c;
}

}  // namespace

GEMM_API gemm_status_t gemm_tune(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void *A,
                                 int64_t lda, const void *B, int64_t ldb, void *C, int64_t ldc,
                                 gemm_dtype_t in_dtype, gemm_dtype_t out_dtype,
                                 gemm_precision_t precision_mode, gemm_layout_t a_layout,
                                 gemm_layout_t b_layout, void *cuda_stream, int32_t iters,
                                 gemm_tune_result_t *result) {
  if (!h || iters < 1 || iters > 1000) return GEMM_ERR_INVALID_ARG;
  const Problem P{M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, precision_mode, a_layout,
                  b_layout};
  const Options base = options_of(h);
  Plan pl0;
  gemm_status_t st = make_plan(P, base, h->sm_count, &pl0);
  if (st != GEMM_OK) return st;
  DeviceGuard g(h->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  // Candidates: the untuned plan first, then every combination of the tile-shape options
  // that plans to a distinct configuration.
  struct Cand {
    Options o;
    Plan pl;
  };
  std::vector<Cand> cands{{base, pl0}};
  if (pl0.info.path == GEMM_PATH_TCGEN05) {
    for (int pair : {1, 2})
      for (int bn : {128, 256})
        for (int sk : {1, 2})
          for (int kps : {1, 2})
            for (int gm : {4, 8, 16}) {
              Options o = base;
              o.cta_pair = pair, o.block_n = bn, o.stream_k = sk, o.stage_k = kps, o.group_m = gm;
              Plan pl;
              if (make_plan(P, o, h->sm_count, &pl) != GEMM_OK) continue;
              const gemm_tune_result_t c = choice_of(o, pl);
              bool dup = false;
              for (const Cand &x : cands) {
                const gemm_tune_result_t d = choice_of(x.o, x.pl);
                // two plans differ if their tiles, stage width, raster group or split differ
                dup |= d.cta_pair == c.cta_pair && d.block_n == c.block_n &&
                       d.stage_k == c.stage_k && d.group_m == c.group_m &&
                       (x.pl.info.split_tiles > 0) == (pl.info.split_tiles > 0);
              }
              if (!dup) cands.push_back({o, pl});
            }
  }
  cudaEvent_t e0 = nullptr, e1 = nullptr;
  if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess) {
    if (e0) cudaEventDestroy(e0);
    cudaGetLastError();
    return GEMM_ERR_CUDA;
  }
  float best = 0.0f, first = 0.0f;
  size_t best_i = 0;
  for (size_t i = 0; i < cands.size() && st == GEMM_OK; ++i) {
    st = execute(h, P, cands[i].pl, s);  // warm-up: workspaces sized, code loaded
    for (int r = 0; r < iters && st == GEMM_OK; ++r) {
      if (r == 0 && cudaEventRecord(e0, s) != cudaSuccess) st = GEMM_ERR_CUDA;
      if (st == GEMM_OK) st = execute(h, P, cands[i].pl, s);
    }
    float ms = 0.0f;
    if (st == GEMM_OK && (cudaEventRecord(e1, s) != cudaSuccess ||
                          cudaEventSynchronize(e1) != cudaSuccess ||
                          cudaEventElapsedTime(&ms, e0, e1) != cudaSuccess))
      st = GEMM_ERR_CUDA;
    const float us = ms * 1000.0f / static_cast<float>(iters);
    if (i == 0) first = us;
    if (st == GEMM_OK && (i == 0 || us < best)) best = us, best_i = i;
  }
  cudaEventDestroy(e0);
  cudaEventDestroy(e1);
  if (st != GEMM_OK) {
    cudaGetLastError();
    return st;
  }
  gemm_tune_result_t r = choice_of(cands[best_i].o, cands[best_i].pl);
  r.candidates = static_cast<int32_t>(cands.size());
  r.best_us = best;
  r.default_us = first;
  TuneEntry t{M, N, K, in_dtype, out_dtype, precision_mode, a_layout, b_layout, r};
  bool replaced = false;
  for (TuneEntry &x : h->tuned)
    if (x.M == M && x.N == N && x.K == K && x.in_dtype == in_dtype && x.out_dtype == out_dtype &&
        x.precision == precision_mode && x.a_layout == a_layout && x.b_layout == b_layout)
      x = t, replaced = true;
  if (!replaced) h->tuned.push_back(t);
  if (result) *result = r;
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_tune_clear(gemm_handle_t h) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  h->tuned.clear();
  return GEMM_OK;
}

// ------------------------------------------------------------------ row softmax

GEMM_API gemm_status_t gemm_softmax_rows(gemm_handle_t h, int64_t M, int64_t N, const void *X,
                                         int64_t ldx, void *Y, int64_t ldy, gemm_dtype_t in_dtype,
                                         gemm_dtype_t out_dtype, void *cuda_stream) {
  if (!h || M < 0 || N < 0) return GEMM_ERR_INVALID_ARG;
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return GEMM_ERR_INVALID_ARG;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!X || !Y || ldx < N || ldy < N) return GEMM_ERR_INVALID_ARG;
  if (M > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
  const int ies = esize_of(in_dtype), oes = esize_of(out_dtype);
  if (reinterpret_cast<uintptr_t>(X) % ies || reinterpret_cast<uintptr_t>(Y) % oes)
    return GEMM_ERR_ALIGNMENT;
  // In place is allowed (the homework's kernel overwrites its input); any other overlap
  // is not.
  const bool in_place = X == Y && ldx == ldy && in_dtype == out_dtype;
  uintptr_t xl, xh, yl, yh;
  span_of(X, M, N, ldx, GEMM_ROW_MAJOR, ies, &xl, &xh);
  span_of(Y, M, N, ldy, GEMM_ROW_MAJOR, oes, &yl, &yh);
  if (!in_place && xl < yh && yl < xh) return GEMM_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  const cudaError_t e = softmax_rows_launch(X, ldx, in_dtype, Y, ldy, out_dtype, M, N, h->sm_count,
                                            static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "softmax launch");
  h->launches += 1;
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_run(gemm_handle_t h, int64_t M, int64_t N, int64_t K, const void *A,
                                int64_t lda, const void *B, int64_t ldb, void *C, int64_t ldc,
                                gemm_dtype_t in_dtype, gemm_dtype_t out_dtype,
                                gemm_precision_t precision_mode) {
  return gemm_run_ex(h, M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, precision_mode,
                     GEMM_ROW_MAJOR, GEMM_ROW_MAJOR, nullptr);
}

namespace {

// 2D copy of `rows` lines of `width` bytes between pitched buffers.
cudaError_t copy2d(void *dst, size_t dpitch, const void *src, size_t spitch, size_t width,
                   size_t rows, cudaMemcpyKind kind, cudaStream_t s) {
  if (rows == 0 || width == 0) return cudaSuccess;
  return cudaMemcpy2DAsync(dst, dpitch, src, spitch, width, rows, kind, s);
}

// Splits [0, extent) into copy panels, writing their starts and the end to start[] and
// returning their number: panels of width w (`width`, else about extent/6, at least 1024; a
// multiple of 256, the CTA-pair tile) while more than two remain, then halves down to 256, so
// that the last product and the last copy out, which nothing overlaps, are short.
int host_panels(int64_t extent, int64_t width, int64_t *start) {
  constexpr int kMax = gemm_handle_s::kMaxPanels;
  int64_t w = width;
  if (w == 0) w = round_up((extent + 5) / 6, 256) < 1024 ? 1024 : round_up((extent + 5) / 6, 256);
  if ((extent + w - 1) / w > kMax / 2) w = round_up((extent + kMax / 2 - 1) / (kMax / 2), 256);
  int n = 0;
  for (int64_t x = 0; x < extent; ++n) {
    const int64_t left = extent - x;
    int64_t len = left > 2 * w ? w : left <= 256 ? left : round_up(left / 2, 256);
    if (n == kMax - 1) len = left;
    start[n] = x;
    x += len;
  }
  start[n] = extent;
  return n;
}

gemm_status_t host_pipeline_setup(gemm_handle_t h) {
  if (h->hp_ready) return GEMM_OK;
  for (cudaStream_t &st : h->hp_stream)
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) return GEMM_ERR_CUDA;
  for (cudaEvent_t &ev : h->hp_event)
    if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) return GEMM_ERR_CUDA;
  h->hp_ready = true;
  return GEMM_OK;
}

}  // namespace

namespace {

// ------------------------------------------------------------ six-stride interface
//
// "Chapter 13: The Blocked Matmul Kernel", section 13.4: the host wrapper passes the
// kernel both strides of A, B and C, so any 2D view is an operand. Views with a unit stride
// and a leading stride that spans a whole line are read (or written) in place through the
// layout path; a column-major C is produced as C^T = B^T A^T into its storage read as a
// row-major N x M matrix (a transposed operand is the same storage with the other layout,
// as in "Triton from zero, Lesson 4", homework 2); any other view is gathered into a
// handle-owned buffer first, and any other C is written to a row-major temporary and
// scattered.

struct StridedPlan {
  Problem P;             // the problem the planner sees (pointers into st_buf where gathered)
  bool gather_a, gather_b;
  int c_mode;            // gemm_strided_info_t::c_mode
  const void *src_a, *src_b;
  int64_t sa0, sa1, sb0, sb1;  // strides of the planner's A (M' x K) and B (K x N') sources
  int64_t da0, da1, db0, db1;  // strides of their gathered copies
  int64_t scm, scn;      // caller's C strides
  void *user_c;
  int64_t c_ld;          // row-major temporary (c_mode 2)
  size_t a_off, b_off, c_off, bytes;
};

// Elements a view spans: (n0 - 1) * s0 + (n1 - 1) * s1 + 1 (0 when empty).
int64_t view_span(int64_t n0, int64_t s0, int64_t n1, int64_t s1) {
  if (n0 <= 0 || n1 <= 0) return 0;
  return (n0 - 1) * s0 + (n1 - 1) * s1 + 1;
}

// Whether a rows x cols view with strides (sr, sc) is a row- or column-major matrix with
// some leading dimension (each line one stride apart, lines not overlapping).
bool view_layout(int64_t rows, int64_t cols, int64_t sr, int64_t sc, int *layout, int64_t *ld) {
  const int64_t r1 = rows > 1 ? rows : 1, c1 = cols > 1 ? cols : 1;
  if ((sc == 1 || cols <= 1) && (rows <= 1 || sr >= c1)) {
    *layout = GEMM_ROW_MAJOR;
    *ld = rows <= 1 ? c1 : sr;
    return true;
  }
  if ((sr == 1 || rows <= 1) && (cols <= 1 || sc >= r1)) {
    *layout = GEMM_COL_MAJOR;
    *ld = cols <= 1 ? r1 : sc;
    return true;
  }
  return false;
}

// Placeholder base for buffers that exist only once the call runs (planning only): a low
// address no device allocation uses, 256-byte aligned like the real buffer.
char *const kPlanBase = reinterpret_cast<char *>(static_cast<uintptr_t>(256));

gemm_status_t make_strided_plan(int64_t M, int64_t N, int64_t K, const void *A, int64_t sam,
                                int64_t sak, const void *B, int64_t sbk, int64_t sbn, void *C,
                                int64_t scm, int64_t scn, int in_dtype, int out_dtype,
                                int precision, char *buf, StridedPlan *out) {
  StridedPlan S{};
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (!valid_dtype(in_dtype) || !valid_dtype(out_dtype)) return GEMM_ERR_INVALID_ARG;
  const int es = esize_of(in_dtype), os = esize_of(out_dtype);
  S.user_c = C;
  S.scm = scm, S.scn = scn;
  if (M == 0 || N == 0) {  // nothing is written: a valid empty problem for the planner
    S.P = Problem{M, N, K, A, 1, B, 1, C, 1, in_dtype, out_dtype, precision, GEMM_ROW_MAJOR,
                  GEMM_ROW_MAJOR};
    S.P.lda = K > 1 ? K : 1, S.P.ldb = N > 1 ? N : 1, S.P.ldc = N > 1 ? N : 1;
    *out = S;
    return GEMM_OK;
  }
  if (sam < 0 || sak < 0 || sbk < 0 || sbn < 0) return GEMM_ERR_INVALID_ARG;
  if ((M > 1 && scm < 1) || (N > 1 && scn < 1)) return GEMM_ERR_INVALID_ARG;
  if (M > 1 && N > 1) {  // no two elements of C may share an address
    const bool n_inner = scn <= scm;
    const int64_t s_in = n_inner ? scn : scm, e_in = n_inner ? N : M;
    const int64_t s_out = n_inner ? scm : scn;
    if (s_out < s_in * (e_in - 1) + 1) return GEMM_ERR_INVALID_ARG;
  }
  if (!C) return GEMM_ERR_INVALID_ARG;
  if (K > 0 && (!A || !B)) return GEMM_ERR_INVALID_ARG;
  // C may not overlap what the product reads.
  const uintptr_t c_lo = reinterpret_cast<uintptr_t>(C);
  const uintptr_t c_hi = c_lo + static_cast<uintptr_t>(view_span(M, scm, N, scn) * os);
  if (K > 0) {
    const uintptr_t a_lo = reinterpret_cast<uintptr_t>(A), b_lo = reinterpret_cast<uintptr_t>(B);
    const uintptr_t a_hi = a_lo + static_cast<uintptr_t>(view_span(M, sam, K, sak) * es);
    const uintptr_t b_hi = b_lo + static_cast<uintptr_t>(view_span(K, sbk, N, sbn) * es);
    if ((c_lo < a_hi && a_lo < c_hi) || (c_lo < b_hi && b_lo < c_hi)) return GEMM_ERR_INVALID_ARG;
  }
  // C: row-major in place; column-major in place as C^T = B^T A^T; else a temporary.
  int c_layout = 0;
  int64_t ldc = 0;
  int64_t Mp = M, Np = N;
  S.src_a = A, S.sa0 = sam, S.sa1 = sak;
  S.src_b = B, S.sb0 = sbk, S.sb1 = sbn;
  if (view_layout(M, N, scm, scn, &c_layout, &ldc) && c_layout == GEMM_ROW_MAJOR) {
    S.c_mode = 0;
  } else if (view_layout(M, N, scm, scn, &c_layout, &ldc)) {
    S.c_mode = 1;
    Mp = N, Np = M;
    S.src_a = B, S.sa0 = sbn, S.sa1 = sbk;  // A' = B^T: A'(i, k) = B(k, i)
    S.src_b = A, S.sb0 = sak, S.sb1 = sam;  // B' = A^T: B'(k, j) = A(j, k)
  } else {
    S.c_mode = 2;
  }
  size_t cursor = 0;
  auto take = [&](int64_t elems, int esz) {
    const size_t off = cursor;
    cursor = static_cast<size_t>(round_up(static_cast<int64_t>(cursor) + elems * esz, 256));
    return off;
  };
  int a_layout = GEMM_ROW_MAJOR, b_layout = GEMM_ROW_MAJOR;
  int64_t lda = 1, ldb = 1;
  const void *pa = S.src_a, *pb = S.src_b;
  if (K > 0 && !view_layout(Mp, K, S.sa0, S.sa1, &a_layout, &lda)) {
    S.gather_a = true;  // row-major copy: A'(i, k) at i * lda + k
    a_layout = GEMM_ROW_MAJOR;
    lda = round_up(K, 16 / es);
    S.da0 = lda, S.da1 = 1;
    S.a_off = take(Mp * lda, es);
    pa = buf + S.a_off;
  }
  if (K > 0 && !view_layout(K, Np, S.sb0, S.sb1, &b_layout, &ldb)) {
    S.gather_b = true;  // column-major copy (K-major, what the MMA reads best): B'(k, j) at j * ldb + k
    b_layout = GEMM_COL_MAJOR;
    ldb = round_up(K, 16 / es);
    S.db0 = 1, S.db1 = ldb;
    S.b_off = take(Np * ldb, es);
    pb = buf + S.b_off;
  }
  if (K == 0) lda = K > 1 ? K : 1, ldb = Np > 1 ? Np : 1;
  void *pc = C;
  if (S.c_mode == 2) {
    S.c_ld = round_up(N, 16 / os);
    ldc = S.c_ld;
    S.c_off = take(M * S.c_ld, os);
    pc = buf + S.c_off;
  }
  S.bytes = cursor;
  S.P = Problem{Mp, Np, K, pa, lda, pb, ldb, pc, ldc, in_dtype, out_dtype, precision, a_layout,
                b_layout};
  *out = S;
  return GEMM_OK;
}

}  // namespace

GEMM_API gemm_status_t gemm_plan_strided(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                         const void *A, int64_t stride_am, int64_t stride_ak,
                                         const void *B, int64_t stride_bk, int64_t stride_bn,
                                         void *C, int64_t stride_cm, int64_t stride_cn,
                                         gemm_dtype_t in_dtype, gemm_dtype_t out_dtype,
                                         gemm_precision_t precision_mode, int32_t sm_count,
                                         gemm_plan_info_t *info, gemm_strided_info_t *sinfo) {
  StridedPlan S;
  gemm_status_t st = make_strided_plan(M, N, K, A, stride_am, stride_ak, B, stride_bk, stride_bn,
                                       C, stride_cm, stride_cn, in_dtype, out_dtype,
                                       precision_mode, kPlanBase, &S);
  if (st != GEMM_OK) return st;
  Plan pl;
  st = make_plan(S.P, options_for(h, S.P), sm_count, &pl);
  if (st != GEMM_OK) return st;
  if (info) *info = pl.info;
  if (sinfo) {
    sinfo->a_gathered = S.gather_a;
    sinfo->b_gathered = S.gather_b;
    sinfo->c_mode = S.c_mode;
    sinfo->buffer_bytes = static_cast<int64_t>(S.bytes);
  }
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_run_strided(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                        const void *A, int64_t stride_am, int64_t stride_ak,
                                        const void *B, int64_t stride_bk, int64_t stride_bn,
                                        void *C, int64_t stride_cm, int64_t stride_cn,
                                        gemm_dtype_t in_dtype, gemm_dtype_t out_dtype,
                                        gemm_precision_t precision_mode, void *cuda_stream) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  StridedPlan S;
  gemm_status_t st = make_strided_plan(M, N, K, A, stride_am, stride_ak, B, stride_bk, stride_bn,
                                       C, stride_cm, stride_cn, in_dtype, out_dtype,
                                       precision_mode, kPlanBase, &S);
  if (st != GEMM_OK) return st;
  Plan pl;
  st = make_plan(S.P, options_for(h, S.P), h->sm_count, &pl);  // argument checks before any work
  if (st != GEMM_OK || pl.info.path == GEMM_PATH_NONE) return st;
  DeviceGuard g(h->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(cuda_stream);
  if (S.bytes > h->st_bytes) {
    if (h->st_buf) cudaFree(h->st_buf);  // synchronises: no launched work still uses it
    h->st_buf = nullptr;
    h->st_bytes = 0;
    if (cudaMalloc(&h->st_buf, S.bytes) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_NO_MEMORY;
    }
    h->st_bytes = S.bytes;
  }
  // the same plan with the real buffer
  st = make_strided_plan(M, N, K, A, stride_am, stride_ak, B, stride_bk, stride_bn, C, stride_cm,
                         stride_cn, in_dtype, out_dtype, precision_mode,
                         static_cast<char *>(h->st_buf), &S);
  if (st == GEMM_OK) st = make_plan(S.P, options_for(h, S.P), h->sm_count, &pl);
  if (st != GEMM_OK) return st;
  const int es = esize_of(in_dtype), os = esize_of(out_dtype);
  cudaError_t e;
  if (S.gather_a) {
    e = strided_copy_launch(S.src_a, S.sa0, S.sa1, const_cast<void *>(S.P.A), S.da0, S.da1,
                            S.P.M, S.P.K, es, s);
    if (e != cudaSuccess) return cuda_fail(e, "gather A");
    h->launches += 1;
  }
  if (S.gather_b) {
    e = strided_copy_launch(S.src_b, S.sb0, S.sb1, const_cast<void *>(S.P.B), S.db0, S.db1,
                            S.P.K, S.P.N, es, s);
    if (e != cudaSuccess) return cuda_fail(e, "gather B");
    h->launches += 1;
  }
  st = execute(h, S.P, pl, s);
  if (st != GEMM_OK) return st;
  if (S.c_mode == 2) {
    e = strided_copy_launch(S.P.C, S.c_ld, 1, S.user_c, S.scm, S.scn, M, N, os, s);
    if (e != cudaSuccess) return cuda_fail(e, "scatter C");
    h->launches += 1;
  }
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_run_host(gemm_handle_t h, int64_t M, int64_t N, int64_t K,
                                     const void *A, int64_t lda, const void *B, int64_t ldb,
                                     void *C, int64_t ldc, gemm_dtype_t in_dtype,
                                     gemm_dtype_t out_dtype, gemm_precision_t precision_mode,
                                     gemm_layout_t a_layout, gemm_layout_t b_layout,
                                     void *cuda_stream) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  const Problem HP{M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, precision_mode, a_layout,
                   b_layout};
  gemm_status_t st = check_args(HP);
  if (st != GEMM_OK) return st;
  DeviceGuard g(h->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  cudaStream_t user = static_cast<cudaStream_t>(cuda_stream);
  if (M == 0 || N == 0) return GEMM_OK;
  const int es = esize_of(in_dtype), os = esize_of(out_dtype);
  const int64_t align_e = 16 / es, align_o = 16 / os;
  // Device copies with 16-byte aligned leading dimensions (TMA-legal in place).
  const bool a_row = a_layout == GEMM_ROW_MAJOR, b_row = b_layout == GEMM_ROW_MAJOR;
  const int64_t a_outer = a_row ? M : K, a_inner = a_row ? K : M;
  const int64_t b_outer = b_row ? K : N, b_inner = b_row ? N : K;
  const int64_t lda_d = round_up(a_inner > 0 ? a_inner : 1, align_e);
  const int64_t ldb_d = round_up(b_inner > 0 ? b_inner : 1, align_e);
  const int64_t ldc_d = round_up(N, align_o);
  const size_t a_bytes = static_cast<size_t>(round_up(a_outer * lda_d * es, 256));
  const size_t b_bytes = static_cast<size_t>(round_up(b_outer * ldb_d * es, 256));
  const size_t c_bytes = static_cast<size_t>(M * ldc_d * os);
  st = host_pipeline_setup(h);
  if (st != GEMM_OK) return st;
  if (a_bytes + b_bytes + c_bytes > h->hp_bytes) {
    // earlier calls may still copy from or into the old buffer
    for (cudaStream_t hs : h->hp_stream) cudaStreamSynchronize(hs);
    if (h->hp_buf) cudaFree(h->hp_buf);
    h->hp_buf = nullptr;
    h->hp_bytes = 0;
    if (cudaMalloc(&h->hp_buf, a_bytes + b_bytes + c_bytes) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_NO_MEMORY;
    }
    h->hp_bytes = a_bytes + b_bytes + c_bytes;
  }
  char *dA = static_cast<char *>(h->hp_buf);
  char *dB = dA + a_bytes;
  char *dC = dB + b_bytes;
  const char *hA = static_cast<const char *>(A), *hB = static_cast<const char *>(B);
  char *hC = static_cast<char *>(C);

  // The copies in alternate between row panels of A and column panels of B (A first). Each
  // arriving panel completes the C block that pairs it with every panel of the other operand
  // already on the device; that block is multiplied (one product over the full K) and copied
  // out while later panels copy in, so the copy out starts after two panels instead of after
  // all of B.
  int64_t a_start[gemm_handle_s::kMaxPanels + 1], b_start[gemm_handle_s::kMaxPanels + 1];
  const int na = host_panels(M, h->host_panel, a_start);
  const int nb = host_panels(N, h->host_panel, b_start);
  cudaStream_t s_in = h->hp_stream[0], s_mm = h->hp_stream[1], s_out = h->hp_stream[2];
  cudaEvent_t e_start = h->hp_event[0], e_done = h->hp_event[1];
  cudaEvent_t *e_in = h->hp_event + 2, *e_mm = h->hp_event + 2 + 2 * gemm_handle_s::kMaxPanels;
  cudaError_t e = cudaEventRecord(e_start, user);
  for (cudaStream_t hs : h->hp_stream)
    if (e == cudaSuccess) e = cudaStreamWaitEvent(hs, e_start, 0);
  if (e != cudaSuccess) return cuda_fail(e, "host pipeline: start");
  int ia = 0, ib = 0;  // panels of A and of B on the device
  for (int step = 0; ia < na || ib < nb; ++step) {
    const bool take_a = ia < na && (ib >= nb || ia <= ib);
    int64_t r0, rows, c0, cols;  // the C block this panel completes
    if (take_a) {
      r0 = a_start[ia];
      rows = a_start[ia + 1] - r0;
      c0 = 0;
      cols = b_start[ib];
      if (K > 0)
        e = a_row ? copy2d(dA + r0 * lda_d * es, lda_d * es, hA + r0 * lda * es, lda * es, K * es,
                           rows, cudaMemcpyHostToDevice, s_in)
                  : copy2d(dA + r0 * es, lda_d * es, hA + r0 * es, lda * es, rows * es, K,
                           cudaMemcpyHostToDevice, s_in);
      ++ia;
    } else {
      c0 = b_start[ib];
      cols = b_start[ib + 1] - c0;
      r0 = 0;
      rows = a_start[ia];
      if (K > 0)
        e = b_row ? copy2d(dB + c0 * es, ldb_d * es, hB + c0 * es, ldb * es, cols * es, K,
                           cudaMemcpyHostToDevice, s_in)
                  : copy2d(dB + c0 * ldb_d * es, ldb_d * es, hB + c0 * ldb * es, ldb * es,
                           K * es, cols, cudaMemcpyHostToDevice, s_in);
      ++ib;
    }
    if (e != cudaSuccess) return cuda_fail(e, "host pipeline: copy in");
    if (rows == 0 || cols == 0) continue;  // nothing of the other operand yet
    if ((e = cudaEventRecord(e_in[step], s_in)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s_mm, e_in[step], 0)) != cudaSuccess)
      return cuda_fail(e, "host pipeline: order");
    const char *a_blk = a_row ? dA + r0 * lda_d * es : dA + r0 * es;
    const char *b_blk = b_row ? dB + c0 * es : dB + c0 * ldb_d * es;
    char *c_blk = dC + (r0 * ldc_d + c0) * os;
    const Problem P{rows, cols, K, a_blk, lda_d, b_blk, ldb_d, c_blk, ldc_d,
                    in_dtype, out_dtype, precision_mode, a_layout, b_layout};
    Plan pl;
    st = make_plan(P, options_for(h, P), h->sm_count, &pl);
    if (st != GEMM_OK) return st;
    st = execute(h, P, pl, s_mm);
    if (st != GEMM_OK) return st;
    if ((e = cudaEventRecord(e_mm[step], s_mm)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(s_out, e_mm[step], 0)) != cudaSuccess ||
        (e = copy2d(hC + (r0 * ldc + c0) * os, ldc * os, c_blk, ldc_d * os, cols * os, rows,
                    cudaMemcpyDeviceToHost, s_out)) != cudaSuccess)
      return cuda_fail(e, "host pipeline: copy out");
  }
  if ((e = cudaEventRecord(e_done, s_out)) != cudaSuccess ||
      (e = cudaStreamWaitEvent(user, e_done, 0)) != cudaSuccess)
    return cuda_fail(e, "host pipeline: join");
  return GEMM_OK;
}

GEMM_API gemm_status_t gemm_get_status(gemm_handle_t h, void *cuda_stream) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  DeviceGuard g(h->device);
  if (!g.ok) return GEMM_ERR_CUDA;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(cuda_stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  int word = 0;
  e = cudaMemcpy(&word, h->status, sizeof word, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "read status word");
  if (word != 0) {
    e = cudaMemset(h->status, 0, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e, "clear status word");
    return static_cast<gemm_status_t>(word);
  }
  return GEMM_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot call cudaMalloc at the point where they need a product: code that
// runs while a framework owns every device allocation (a plugin inside another runtime's
// memory pool), deployments that reserve all device memory up front and forbid growth,
// and host callbacks or real-time paths where a cudaMalloc (which may synchronise the
// device) is not allowed. gemm_run_noalloc serves them without a handle: the staging
// copies that misaligned operands and MN-major tf32 operands need go to a fixed, file-scope
// device array instead of a workspace that grows on demand.
namespace {

constexpr size_t kStaticStatusBytes = 256;  // first 256 bytes: the call's status word
static_assert(GEMM_NOALLOC_SCRATCH_BYTES > kStaticStatusBytes, "scratch too small");

// Every GPU on which this library's device code is loaded keeps this array until the
// process exits. All calls on a device share it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];  // device address of g_noalloc_scratch, per device
int g_noalloc_sms[kMaxDevices];

// Per-device set-up, done by the first call on each device with that device current:
// look up the array's device address (host code only has a stand-in symbol for it) and
// the SM count. Later calls reuse both.
gemm_status_t noalloc_setup(int dev, void **scratch, int *sms) {
  if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    int major = 0, minor = 0, count = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      cudaGetLastError();
      return GEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_DEVICE;
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) return cuda_fail(e, "look up the static scratch");
    g_noalloc_sms[dev] = count;
    g_noalloc_ptr[dev] = p;
  }
  *scratch = g_noalloc_ptr[dev];
  *sms = g_noalloc_sms[dev];
  return GEMM_OK;
}

// Same launches as the handle path, with the staging area and the status word taken
// from the static scratch (or the caller's status word) and default options.
gemm_status_t execute_noalloc(void *scratch, int *status, const Problem &P, const Plan &pl,
                              cudaStream_t s) {
  const gemm_plan_info_t &I = pl.info;
  cudaError_t e;
  switch (I.path) {
    case GEMM_PATH_NONE: return GEMM_OK;
    case GEMM_PATH_ZERO_FILL:
      e = zero_fill_launch(P.C, P.ldc, P.M, P.N, P.out_dtype, s);
      return e == cudaSuccess ? GEMM_OK : cuda_fail(e, "zero fill launch");
    case GEMM_PATH_FMA: {
      FmaParams fp{P.M, P.N, P.K, P.A, P.lda, P.B, P.ldb, P.C, P.ldc, P.in_dtype, P.out_dtype,
                   P.a_layout == GEMM_COL_MAJOR, P.b_layout == GEMM_COL_MAJOR, pl.acc_chunk};
      e = fma_launch(fp, pl.fma_tile, s);
      return e == cudaSuccess ? GEMM_OK : cuda_fail(e, "fma launch");
    }
    default: break;
  }
  const size_t limit = GEMM_NOALLOC_SCRATCH_BYTES - kStaticStatusBytes;
  if (static_cast<size_t>(I.workspace_bytes) > limit) {
    if (log_enabled())
      std::fprintf(stderr, "[gemm] gemm_run_noalloc: staging needs %lld bytes, limit %zu\n",
                   static_cast<long long>(I.workspace_bytes), limit);
    return GEMM_ERR_UNSUPPORTED;
  }
  char *staging = static_cast<char *>(scratch) + kStaticStatusBytes;
  if (!status) {
    // The static status word keeps the last call's value: clear it for this call.
    status = static_cast<int *>(scratch);
    e = cudaMemsetAsync(status, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_fail(e, "clear the static status word");
  }
  const int es = esize_of(P.in_dtype);
  const void *a_ptr = pl.a.ptr;
  int64_t a_ld = pl.a.ld;
  const void *b_ptr = pl.b.ptr;
  int64_t b_ld = pl.b.ld;
  for (const OperandPlan *o : {&pl.a, &pl.b}) {
    if (!o->staged) continue;
    void *dst = staging + o->ws_offset;
    e = stage_operand(*o, dst, es, s);
    if (e != cudaSuccess) return cuda_fail(e, "stage operand");
    if (o == &pl.a)
      a_ptr = dst, a_ld = o->staged_ld;
    else
      b_ptr = dst, b_ld = o->staged_ld;
  }
  const Options defaults;
  return launch_tc(P, pl, a_ptr, a_ld, b_ptr, b_ld, status, gemm_handle_s().timeout_us * 1000ull,
                   defaults.group_m, 0, SplitK(), s);
}

}  // namespace

extern "C" GEMM_API gemm_status_t gemm_run_noalloc(
    int64_t M, int64_t N, int64_t K, const void *A, int64_t lda, const void *B, int64_t ldb,
    void *C, int64_t ldc, gemm_dtype_t in_dtype, gemm_dtype_t out_dtype,
    gemm_precision_t precision_mode, gemm_layout_t a_layout, gemm_layout_t b_layout,
    int *device_status, void *cuda_stream) {
  const Problem P{M, N, K, A, lda, B, ldb, C, ldc, in_dtype, out_dtype, precision_mode, a_layout,
                  b_layout};
  Plan pl;
  gemm_status_t st = check_args(P);
  if (st != GEMM_OK) return st;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return GEMM_ERR_DEVICE;
  }
  void *scratch = nullptr;
  int sms = 0;
  st = noalloc_setup(dev, &scratch, &sms);
  if (st != GEMM_OK) return st;
  st = make_plan(P, Options(), sms, &pl);
  if (st != GEMM_OK) return st;
  if (pl.info.path == GEMM_PATH_TCGEN05_3XTF32 &&
      static_cast<size_t>(pl.info.workspace_bytes) > GEMM_NOALLOC_SCRATCH_BYTES - kStaticStatusBytes) {
    // Exact fp32 whose split operands do not fit the array: the fp32 FMA kernel needs none.
    Options fma;
    fma.force_path = 2;
    st = make_plan(P, fma, sms, &pl);
    if (st != GEMM_OK) return st;
  }
  return execute_noalloc(scratch, device_status, P, pl, static_cast<cudaStream_t>(cuda_stream));
}
