// tune.cu -- gemm_tune / gemm_tune_clear: measured per-signature choices of the planner's
// tile-shape options, kept on the handle.
#include <vector>

#include "api_internal.h"

using namespace gemm_gb300;
using namespace gemm_gb300::api;

extern "C" {

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
  c.tile_rows = pl.cta_rows;
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
    // Shorter pair tiles (96 rows per CTA) only for bandwidth-bound products (under ~256
    // flops per byte of A, B and C), where they can even out the rounds.
    const std::vector<int> rows_set =
        intensity_of(P) < kBandwidthBound ? std::vector<int>{0, 96} : std::vector<int>{0};
    for (int pair : {1, 2})
      for (int bn : {128, 256})
        for (int sk : {1, 2})
          for (int kps : {1, 2})
            for (int gm : {4, 8, 16})
              for (int rows : rows_set) {
                Options o = base;
                o.cta_pair = pair, o.block_n = bn, o.stream_k = sk, o.stage_k = kps, o.group_m = gm;
                o.tile_rows = rows;
                Plan pl;
                if (make_plan(P, o, h->sm_count, &pl) != GEMM_OK) continue;
                const gemm_tune_result_t c = choice_of(o, pl);
                bool dup = false;
                for (const Cand &x : cands) {
                  const gemm_tune_result_t d = choice_of(x.o, x.pl);
                  // two plans differ if their tiles, stage width, raster group or split differ
                  dup |= d.cta_pair == c.cta_pair && d.block_n == c.block_n &&
                         d.stage_k == c.stage_k && d.group_m == c.group_m &&
                         d.tile_rows == c.tile_rows &&
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
    st = execute(h, P, cands[i].pl, s, false);  // warm-up: workspaces sized, code loaded
    for (int r = 0; r < iters && st == GEMM_OK; ++r) {
      if (r == 0 && cudaEventRecord(e0, s) != cudaSuccess) st = GEMM_ERR_CUDA;
      if (st == GEMM_OK) st = execute(h, P, cands[i].pl, s, false);
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

}  // extern "C"
