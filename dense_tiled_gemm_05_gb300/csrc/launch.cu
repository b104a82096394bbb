// launch.cu -- from a plan to kernel launches: tensor-map encoding, instruction
// descriptors, the handle's workspaces (staged operands, split-K partials and flags), and
// the launch of the planned kernel.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "api_internal.h"

using namespace gemm_gb300;
using namespace gemm_gb300::api;

namespace gemm_gb300 {
namespace api {

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

// cuTensorMapEncodeTiled, fetched from the driver through the runtime so the library
// needs no link-time dependency on libcuda.
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
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

static CUtensorMapDataType tmap_dtype(int dt) {
  switch (dt) {
    case GEMM_F16: return CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    case GEMM_BF16: return CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    default: return CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
  }
}

// 2D tensor map: dims {inner, outer}, row pitch ld elements, box {box_inner, box_outer},
// 128-byte swizzle (of 16-byte chunks, or of 32-byte atoms with atom32, the form the
// tensor cores read an MN-major tf32 operand in), zero fill outside the tensor.
bool encode_2d(CUtensorMap *m, int dtype, const void *base, int64_t inner, int64_t outer,
               int64_t ld, uint32_t box_inner, uint32_t box_outer, bool atom32) {
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
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  atom32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS && log_enabled())
    std::fprintf(stderr, "[gemm] cuTensorMapEncodeTiled failed (%d)\n", static_cast<int>(r));
  return r == CUDA_SUCCESS;
}

// 3D tensor map over an MN-major operand that loads a CTA's whole slice of a stage with
// one copy: dims {panel, K, MN / panel} (128-byte panels of M or N, K rows of the stage,
// the panel index), strides {ld, panel} in bytes, box {panel, k_rows, panels}. The box
// lands in shared memory panel after panel, each panel k_rows x 128 bytes, which is the
// layout the 2D loads build one panel at a time. Only for an MN extent that is a whole
// number of panels: a 3D box has no bound inside a panel, so a partial last panel would
// read past the operand's rows instead of reading zeros.
bool encode_3d_panels(CUtensorMap *m, int dtype, const void *base, int64_t mn, int64_t k,
                      int64_t ld, uint32_t k_rows, uint32_t panels, bool atom32) {
  EncodeTiledFn fn = encode_fn();
  const int es = esize_of(dtype);
  const int64_t panel = 128 / es;
  if (!fn || mn % panel != 0 || k <= 1) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(panel), static_cast<cuuint64_t>(k),
                              static_cast<cuuint64_t>(mn / panel)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld * es), 128};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(panel), k_rows, panels};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, tmap_dtype(dtype), 3, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE,
                  atom32 ? CU_TENSOR_MAP_SWIZZLE_128B_ATOM_32B : CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS && log_enabled())
    std::fprintf(stderr, "[gemm] cuTensorMapEncodeTiled (3D panels) failed (%d)\n",
                 static_cast<int>(r));
  return r == CUDA_SUCCESS;
}

static uint32_t make_idesc(int in_dtype, bool a_mn, bool b_mn, int n, int m) {
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

static gemm_status_t ensure_workspace(gemm_handle_t h, size_t bytes) {
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

cudaError_t stage_operand(const OperandPlan &o, void *dst, int es, cudaStream_t s) {
  if (o.split_hl)
    return split2_launch(static_cast<const float *>(o.ptr), o.ld, o.k_contig,
                         static_cast<float *>(dst), o.staged_ld, o.rows, o.k, o.split_kp, s);
  if (o.transpose) return transpose_launch(o.ptr, o.ld, dst, o.staged_ld, o.outer, o.inner, es, s);
  return repack_launch(o.ptr, o.ld, dst, o.staged_ld, o.outer, o.inner, es, s);
}

static gemm_status_t ensure_sk_workspace(gemm_handle_t h, size_t bytes, size_t flag_bytes,
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
  // The epoch word, the arrival count and every flag start at 0.
  if (cudaMemsetAsync(p, 0, flag_bytes, s) != cudaSuccess) {
    cudaFree(p);
    return GEMM_ERR_CUDA;
  }
  h->sk_ws = p;
  h->sk_ws_bytes = bytes;
  return GEMM_OK;
}

// Tensor maps, kernel parameters and launch of the tensor-core kernel for operands that
// are already TMA-legal (in place or staged).
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
  const uint32_t cta_rows_a = static_cast<uint32_t>(pl.cta_rows);
  const uint32_t cta_rows_b = pl.variant.pair ? I.tile_n / 2 : I.tile_n;
  const uint32_t a_box_outer = pl.a.mn_major ? row_elems : cta_rows_a;
  const uint32_t b_box_outer = pl.b.mn_major ? row_elems : cta_rows_b;
  if (!encode_2d(&tmA, P.in_dtype, a_ptr, pl.a.k_inner, pl.a.k_outer, a_ld, row_elems,
                 a_box_outer, es == 4 && pl.a.mn_major) ||
      !encode_2d(&tmB, P.in_dtype, b_ptr, pl.b.k_inner, pl.b.k_outer, b_ld, row_elems,
                 b_box_outer, es == 4 && pl.b.mn_major))
    return GEMM_ERR_CUDA;
  // An MN-major operand whose M or N is a whole number of 128-byte panels is loaded with
  // one 3D copy per stage instead of one 2D copy per panel (the loader issues fewer, larger
  // copies; one copy per panel kept a tf32 B of four panels a stage behind the MMAs).
  int32_t mn_3d = 0;
  if (!pl.variant.exact && !pl.variant.f16acc) {
    const uint32_t k_rows = static_cast<uint32_t>(pl.variant.kps) * row_elems;
    CUtensorMap m3;
    if (pl.a.mn_major && pl.cta_rows == kTcBlockM &&
        encode_3d_panels(&m3, P.in_dtype, a_ptr, pl.a.k_inner, pl.a.k_outer, a_ld, k_rows,
                         cta_rows_a / row_elems, es == 4)) {
      tmA = m3;
      mn_3d |= kMn3dA;
    }
    if (pl.b.mn_major && cta_rows_b % row_elems == 0 &&
        encode_3d_panels(&m3, P.in_dtype, b_ptr, pl.b.k_inner, pl.b.k_outer, b_ld, k_rows,
                         cta_rows_b / row_elems, es == 4)) {
      tmB = m3;
      mn_3d |= kMn3dB;
    }
  }
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
  // The MMA shape is fixed by the kernel: 128 rows per CTA (256 for a pair), whatever
  // number of those rows the tile uses.
  const int mma_m = pl.variant.pair ? 2 * kTcBlockM : kTcBlockM;
  if (I.tile_n % 16 != 0 || I.tile_n < 16 || I.tile_n > 256 || pl.cta_rows > kTcBlockM ||
      I.tile_m != (pl.variant.pair ? 2 * pl.cta_rows : kTcBlockM))
    return GEMM_ERR_UNSUPPORTED;
  tp.idesc = make_idesc(P.in_dtype, pl.a.mn_major, pl.b.mn_major, I.tile_n, mma_m);
  tp.out_dtype = P.out_dtype;
  tp.tma_store = I.tma_store;
  tp.C = P.C;
  tp.ldc = P.ldc;
  tp.status = status;
  tp.timeout_ns = timeout_ns;
  tp.debug_flags = debug_flags;
  tp.chunk_steps = pl.chunk_steps;
  tp.cta_rows = pl.cta_rows;
  tp.split_kb = pl.a.split_hl ? static_cast<int32_t>(pl.a.split_kp / 32) : 0;
  tp.mn_3d = mn_3d;
  // An operand that only one tile column (A) or one tile row (B) reads is streamed once:
  // its loads go to L2 as first to evict, and whole tiles then start their K-loops at
  // staggered K-blocks, so that tiles running side by side do not all fetch the same
  // column band of A (addresses one row pitch apart) at once. Measured on bf16
  // 16384 x 128 x 8192: 53.1 us plain, 50.3 us staggered, 50.4 us with evict_first on A,
  // 48.7 us with both. The fp16 accumulator's running total and the exact kernel's chunk
  // sums take K in order, so the chunked kernel never staggers.
  const bool a_once = I.grid_n == 1, b_once = I.grid_m == 1;
  tp.l2_once = (a_once ? kL2OnceA : 0) | (b_once ? kL2OnceB : 0);
  tp.k_rotate = (a_once || b_once) && !pl.variant.exact && !pl.variant.f16acc ? 17 : 0;
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
      // Workspace: [epoch word, arrival count | one flag per epilogue warp of each CTA of
      // the largest grid (8 per CTA) | partial tiles]. The flag region has a fixed size, so
      // a grown workspace never finds partial data where flags are expected.
      const int64_t ctas_max = sk.h->sm_count > grid ? sk.h->sm_count : grid;
      const size_t flag_region =
          static_cast<size_t>(round_up(static_cast<int64_t>((2 + 8 * ctas_max) * sizeof(int)), 256));
      const size_t part_bytes =
          static_cast<size_t>(slots) * 2 * kTcBlockM * pl.variant.block_n * sizeof(float);
      gemm_status_t st = ensure_sk_workspace(sk.h, flag_region + part_bytes, flag_region, s);
      if (st != GEMM_OK) return st;
      tp.sk_epoch_word = static_cast<int *>(sk.h->sk_ws);
      tp.sk_flags = tp.sk_epoch_word + 2;
      tp.sk_partials = reinterpret_cast<float *>(static_cast<char *>(sk.h->sk_ws) + flag_region);
      // partial tiles: rows [worker][cta rank][128], block_n fp32 columns; 32 x 32 boxes
      if (!encode_2d(&tmP, GEMM_F32, tp.sk_partials, pl.variant.block_n,
                     static_cast<int64_t>(slots) * 2 * kTcBlockM, pl.variant.block_n, 32, 32))
        return GEMM_ERR_CUDA;
    }
  }
  const cudaError_t e = tc_launch(pl.variant, tmA, tmB, tmC, tmP, tp, static_cast<int>(grid), s);
  return e == cudaSuccess ? GEMM_OK : cuda_fail(e, "tcgen05 launch");
}

// GEMM_OPT_FAULT_STALL_PRODUCER value -> kernel debug flags: 1, no loads at all; v >= 2,
// the loader of CTA rank (v & 1) stops after v >> 1 stage fills.
static int stall_flags(int v) {
  if (v == 1) return kDebugStallProducer;
  if (v >= 2) return ((v >> 1) << kDebugStallAfterShift) | ((v & 1) ? kDebugStallRank1 : 0);
  return 0;
}

gemm_status_t execute(gemm_handle_t h, const Problem &P, const Plan &pl, cudaStream_t s,
                      bool record_events) {
  const gemm_plan_info_t &I = pl.info;
  cudaError_t e;
  const cudaEvent_t ev0 = record_events ? h->kernel_events[0] : nullptr;
  const cudaEvent_t ev1 = record_events ? h->kernel_events[1] : nullptr;
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
      if (ev0 && (e = cudaEventRecord(ev0, s)) != cudaSuccess)
        return cuda_fail(e, "record the kernel start event");
      e = fma_launch(fp, pl.fma_tile, s);
      if (e != cudaSuccess) return cuda_fail(e, "fma launch");
      h->launches += 1;
      if (ev1 && (e = cudaEventRecord(ev1, s)) != cudaSuccess)
        return cuda_fail(e, "record the kernel end event");
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
  if (ev0 && (e = cudaEventRecord(ev0, s)) != cudaSuccess)
    return cuda_fail(e, "record the kernel start event");
  st = launch_tc(P, pl, a_ptr, a_ld, b_ptr, b_ld, h->status, h->timeout_us * 1000ull,
                 pl.group_m, stall_flags(h->stall_producer), sk, s);
  if (st != GEMM_OK) return st;
  h->launches += 1;
  if (ev1 && (e = cudaEventRecord(ev1, s)) != cudaSuccess)
    return cuda_fail(e, "record the kernel end event");
  return GEMM_OK;
}

}  // namespace api
}  // namespace gemm_gb300
