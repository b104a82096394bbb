// planner.cu -- argument checks and the plan of one product: which path (tensor cores,
// chunked tensor-core kernel, FMA tiles, zero fill), tile shape, staging of each operand,
// split-K share, and the handle options (or gemm_tune's choice) that steer it.
//
// The host wrapper of "Chapter 13: The Blocked Matmul Kernel" (section 13.4,
// 01_tiled_matmul.py) reads M, K from A and N from B, checks that the inner dimensions
// agree, lets the caller own C, and launches a (cdiv(M, BLOCK_M), cdiv(N, BLOCK_N)) grid
// with cdiv(K, BLOCK_K) K-iterations per tile. Here the caller states M, N, K and the
// leading dimensions explicitly, and the planner maps the same tile grid onto a
// persistent schedule over the SMs.
#include <cmath>
#include <cstdint>

#include "api_internal.h"

using namespace gemm_gb300;
using namespace gemm_gb300::api;

namespace gemm_gb300 {
namespace api {

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
static bool tma_legal(const void *p, int64_t ld, int64_t outer, int es) {
  if (reinterpret_cast<uintptr_t>(p) % 16) return false;
  return outer <= 1 || (ld * es) % 16 == 0;
}

static OperandPlan plan_operand(const void *p, int64_t rows, int64_t cols, int64_t ld, int layout,
                                bool k_is_rows_dim, int es, bool force_stage, bool split_hl,
                                bool k_major_only, size_t *ws_cursor) {
  // (k_major_only: the kernel reads this operand K-major only, so an MN-major one is
  // staged transposed)
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
  o.split_hl = split_hl;
  o.transpose = !split_hl && o.mn_major && k_major_only;
  o.staged = split_hl || o.transpose || force_stage || !tma_legal(p, ld, o.outer, es);
  if (o.staged) {
    if (split_hl) {
      o.split_kp = round_up(o.k, 32);  // 32 fp32 = one 128-byte K-block
      o.k_outer = o.rows;
      o.k_inner = 2 * o.split_kp;
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

double intensity_of(const Problem &P) {
  const double es = esize_of(P.in_dtype), os = esize_of(P.out_dtype);
  const double m = static_cast<double>(P.M), n = static_cast<double>(P.N),
               k = static_cast<double>(P.K);
  return 2.0 * m * n * k / (es * (m * k + k * n) + os * m * n);
}

// Tile slots of the CTA-pair kernel: one cluster of two SMs each, under the CTA cap.
static int64_t pair_slots(int sm_count, int max_ctas) {
  int64_t clusters = sm_count > 1 ? sm_count / 2 : 1;
  if (max_ctas > 0 && max_ctas / 2 < clusters) clusters = max_ctas / 2 > 0 ? max_ctas / 2 : 1;
  return clusters;
}

// Whether splitting the last rounds along K pays on GB300 (interleaved measurements of
// bf16 products). The split share is the last whole round plus the partial one, r of a
// round's worth of tiles with 1 < r < 2 (sk_schedule.h); split, those run about 1.1-1.3
// times slower per tile than whole tiles (partial stores, owners' sums), so sharing them
// out beats the two rounds they otherwise take while r is at most 1.6: 2560^2 x 8192
// (r = 1.32) 66.2 against 84.4 us, 4096^3 (1.37) +5.8 %, 5120^3 (1.26) +7.4 %, 8192^3
// (1.47) +3.6 %; 6144^2 x 4096 (1.58) even; 2048 x 4096 x 4096 (1.68) even; 3072^2 x 4096
// (1.89) -7 %. K must be long enough (8192 x 8192 x 2048, 32 K-blocks, -1.6 %), and a
// product with fewer tiles than slots keeps them whole (2048^2 x 8192 -6 %) unless its
// tiles would leave more than half of the slots idle with a long K-loop (128 or more
// K-blocks): one tile's K-loop then sets the time, and sharing it out wins (bf16
// M x 128 x 8192: M = 2048 22.7 against 34.4 us, 4096 24.9 against 35.1, 8192 33.1
// against 35.2; 128 x 4096 x 4096, 64 K-blocks, 27.1 against 24.9). stream_k: 0 by this
// rule, 1 never, 2 whenever the schedule allows. k_blocks counts 128-byte K-blocks.
bool use_split_k(int stream_k, int64_t tiles, int64_t k_blocks, int64_t slots) {
  if (stream_k == 1) return false;
  if (stream_k == 2) return true;
  if (slots <= 0) return false;
  if (2 * tiles <= slots) return k_blocks >= 128;
  if (tiles <= slots || tiles % slots == 0 || k_blocks < 64) return false;
  const int64_t shared = tiles - (tiles / slots - 1) * slots;  // r * slots
  return 10 * shared <= 16 * slots;
}

// Most pieces a tile is split into when its pieces fill otherwise idle clusters. The owner
// adds every other piece's partial in turn, so the best count grows only as the square
// root of the K-loop: about six for 128 K-blocks (bf16 256 x 256 x 8192: 27 us over 4 to 8
// clusters, 127 us over 76; 1024 x 128 x 8192, 4 tiles: 20.8 us over 32 clusters, 29 over
// 76), sixteen for 1024.
static int64_t idle_split_pieces(int64_t k_blocks) {
  const int64_t p = static_cast<int64_t>(std::sqrt(static_cast<double>(k_blocks) / 4.0) + 0.5);
  return p < 2 ? 2 : p;
}

// Short-K products the FMA kernel takes (see make_plan): K and output-size limits.
constexpr int64_t kFmaMaxK = 24;
constexpr int64_t kFmaMaxOutputs = int64_t{1} << 22;

// Tile width by a wave-quantisation cost model: a persistent grid runs
// ceil(tiles / slots) rounds, each as long as one tile. A 128-wide tile has half the
// flops of a 256-wide one but, measured on GB300, takes about 0.8 of its time (0.74 on
// bf16 2048^2 x 8192, 0.82 on 2560^2 x 8192, both split along K; every MMA re-reads its
// 128 x 16 slice of A from shared memory, so narrow MMAs are starved of shared-memory
// bandwidth); it wins only when it fills the machine much better, e.g. when N itself is
// at most 128.
static int pick_block_n(int64_t M, int64_t N, int64_t k_blocks, bool pair, int stream_k, int sm_count) {
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
  return cost(128, 1.6) < cost(256, 1.0) ? 128 : 256;
}

gemm_status_t make_plan(const Problem &P, const Options &opt, int sm_count, Plan *out) {
  gemm_status_t st = check_args(P);
  if (st != GEMM_OK) return st;
  Plan pl{};
  pl.group_m = opt.group_m;
  pl.stream_k = opt.stream_k;
  pl.cta_rows = kTcBlockM;
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
  // A short K with a moderate output also takes the FMA kernel, unless a tensor-core tile
  // shape is asked for: one launch that reads operands of any alignment, where the tensor
  // cores need staging copies for misaligned rows and a launch whose fixed costs dominate.
  // Replayed from CUDA graphs on GB300 (the 216 products of the ragged sweep, average per
  // product): K = 1 4.5 against 8.8 us, K = 17 7.9 against 9.9, but K = 127 34 against
  // 10 (the FMA kernel walks K serially in steps of 8).
  const bool tile_asked = opt.cta_pair != 0 || opt.block_n != 0 || opt.stage_k != 0 ||
                          opt.tile_rows != 0;
  if (!tile_asked && P.K <= kFmaMaxK && P.M * P.N <= kFmaMaxOutputs) use_fma = true;
  if (opt.force_path == 2) use_fma = true;
  if (opt.force_path == 1) {
    if (f16acc && pl.acc_chunk % 16 != 0) return GEMM_ERR_UNSUPPORTED;
    use_fma = false;
  }
  const bool split = exact && !use_fma;
  if (use_fma) {
    pl.fma_tile = (P.M * P.N <= 256 && !f16acc) ? 4 : f16acc ? 8 : 128;
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
  // K-major only: the fp16-accumulator kernel; tf32 operands when the option asks for the
  // transposed copy (by default the tensor cores read MN-major tf32 in place).
  const bool k_major_only = f16acc || (es == 4 && opt.tf32_transpose != 0);
  pl.a = plan_operand(P.A, P.M, P.K, P.lda, P.a_layout, false, es, opt.force_staging != 0, split,
                      k_major_only, &cursor);
  pl.b = plan_operand(P.B, P.K, P.N, P.ldb, P.b_layout, true, es, opt.force_staging != 0, split,
                      k_major_only, &cursor);
  pl.variant.esize = es;
  pl.variant.a_mn = pl.a.mn_major;
  pl.variant.b_mn = pl.b.mn_major;
  const double intensity = intensity_of(P);
  // CTA pairs (256-row tiles on two SMs) halve the shared-memory and L2 traffic per
  // flop; a problem no taller than one 128-row tile keeps single-CTA tiles, and so does a
  // compute-bound one whose 128 x 256 single-CTA tiles all run at once (one round on the
  // SMs) with a short K-loop, where the pair's cross-SM handshakes cost more than they
  // save (bf16 2048^3: 17.1 against 19.0 us); from 64 K-blocks on, pairs win again (bf16
  // 2048^2 x 4096: 27.7 against 29.4 us; 2048^2 x 8192: 46.3 against 53.0). Bandwidth-bound
  // ones keep pairs, for their wide stages. So do products with so few tiles that even
  // 128-wide pair tiles leave more than half of the clusters idle, when K is long: the
  // split-K rule then shares each tile's K-loop out (bf16 1024 x 512 x 8192: 27.5 against
  // 41.3 us on single-CTA tiles; 512 x 1024 x 16384: 34.4 against 78.1; 128 x 128 x 65536:
  // 61.8 against 289).
  const int64_t single_tiles = ((P.M + kTcBlockM - 1) / kTcBlockM) * ((P.N + 255) / 256);
  const int64_t narrow_kb = (P.K + 128 / es - 1) / (128 / es);
  const bool one_round = single_tiles <= sm_count && intensity >= kBandwidthBound && narrow_kb < 64;
  const bool few_tiles = opt.stream_k != 1 && narrow_kb >= 128 &&
                         2 * ((P.M + 255) / 256) * ((P.N + 127) / 128) <= pair_slots(sm_count, opt.max_ctas);
  pl.variant.pair = opt.cta_pair == 2 ||
                    (opt.cta_pair == 0 && ((P.M > kTcBlockM && !one_round) || few_tiles));
  pl.variant.block_n =
      opt.block_n ? opt.block_n
                  : pick_block_n(P.M, P.N, narrow_kb, pl.variant.pair, split ? 1 : opt.stream_k,
                                 sm_count);
  if (split || f16acc) {  // the chunked kernel has one shape: CTA pairs, 256 x 256 tiles
    pl.variant.exact = split;
    pl.variant.f16acc = f16acc;
    pl.variant.pair = true;
    pl.variant.block_n = 256;
  }
  const bool chunked = pl.variant.exact || pl.variant.f16acc;
  // Rows of A per CTA of a pair tile (GEMM_OPT_TILE_ROWS; 128 by default). The MMA is
  // always 128 rows per CTA; a CTA given fewer loads only those (the rest of its
  // shared-memory rows feed accumulator lanes that are never stored). Shorter tiles do not
  // pay by default: on bf16 M x 128 x 8192 the time stays that of one tile's K-loop, set by
  // each SM's stream of A, whether 64 or 74 clusters run (M = 16384: 47.7 us with 256-row
  // tiles, 50.5 us with 224), but two rounds of shorter tiles can beat one and a part
  // (M = 24576: 71.8 us with 192-row tiles, 80.4 us with 256); gemm_tune tries them.
  const bool rows_ok = pl.variant.pair && !chunked && !pl.a.mn_major;
  if (opt.tile_rows && !rows_ok) return GEMM_ERR_UNSUPPORTED;
  if (opt.tile_rows) pl.cta_rows = opt.tile_rows;
  // Two 128-byte K-blocks per stage (CTA-pair kernel, K-major 16-bit operands): each row
  // of A and B is then fetched 256 contiguous bytes at a time. By default only for
  // bandwidth-bound products (under ~256 flops per byte of A, B and C), where it measured
  // +1.5 % on bf16 16384 x 128 x 8192; compute-bound ones keep the deeper ring of one
  // K-block per stage (4096^3 lost 9 % with wide stages). A split-K keeps narrow K-blocks,
  // the finer unit it shares out (one 256 x 256 x 8192 tile: 128 units for 76 clusters
  // rather than 64): a forced one, and the one that shares few tiles out over idle slots.
  const int64_t clusters = pair_slots(sm_count, opt.max_ctas);
  const int64_t pair_tiles = ((P.M + 2 * pl.cta_rows - 1) / (2 * pl.cta_rows)) *
                             ((P.N + pl.variant.block_n - 1) / pl.variant.block_n);
  const bool idle_split = pl.variant.pair && !chunked && 2 * pair_tiles <= clusters &&
                          use_split_k(opt.stream_k, pair_tiles, narrow_kb, clusters);
  const bool wide_ok = pl.variant.pair && !chunked && es == 2 && !pl.a.mn_major && !pl.b.mn_major;
  if (opt.stage_k == 2 && !wide_ok) return GEMM_ERR_UNSUPPORTED;
  pl.variant.kps = opt.stage_k == 2 || (opt.stage_k == 0 && wide_ok && intensity < kBandwidthBound &&
                                        opt.stream_k != 2 && !idle_split)
                       ? 2
                       : 1;
  I.path = split ? GEMM_PATH_TCGEN05_3XTF32 : f16acc ? GEMM_PATH_TCGEN05_F16ACC : GEMM_PATH_TCGEN05;
  I.tile_m = pl.variant.pair ? 2 * pl.cta_rows : kTcBlockM;
  I.tile_n = pl.variant.block_n;
  I.tile_k = pl.variant.kps * 128 / es;
  I.grid_m = (P.M + I.tile_m - 1) / I.tile_m;
  I.grid_n = (P.N + I.tile_n - 1) / I.tile_n;
  // split operands: three products over each part's padded K
  const int64_t k_total = split ? 3 * pl.a.split_kp : P.K;
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
    // (the fp16 accumulator never splits: its running total takes the chunks in order)
    const bool split = !pl.variant.f16acc && use_split_k(opt.stream_k, tiles, I.k_iters, clusters) &&
                       sk_dp_tiles(static_cast<int32_t>(tiles), static_cast<int32_t>(I.k_iters),
                                   static_cast<int32_t>(clusters), true) < tiles;
    // Tiles split over otherwise idle clusters take a limited number of pieces each.
    const int64_t cap = idle_split_pieces(I.k_iters) * tiles;
    const int64_t slots = split && 2 * tiles <= clusters && cap < clusters ? cap : clusters;
    I.ctas = 2 * (split || tiles > clusters ? slots : tiles);
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
    o.tile_rows = h->tile_rows;
    o.tf32_transpose = h->tf32_transpose;
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
    o.tile_rows = t->choice.tile_rows == kTcBlockM ? 0 : t->choice.tile_rows;
  }
  return o;
}

}  // namespace api
}  // namespace gemm_gb300
