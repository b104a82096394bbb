// gemm_api.cu -- the C ABI of include/gemm.h: handle lifecycle, options, the plan query,
// gemm_run / gemm_run_ex, the device status word, and the row softmax entry point. The
// planner (planner.cu) and launcher (launch.cu) do the work; tune.cu, host_path.cu,
// strided.cu and noalloc.cu hold the other entry points.
#include <cstdio>
#include <cstring>

#include "api_internal.h"

using namespace gemm_gb300;
using namespace gemm_gb300::api;

namespace {

const char *kVersion = "0.1.0";

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
  for (cudaStream_t st : h->hp_stream)
    if (st) cudaStreamDestroy(st);
  for (cudaEvent_t ev : h->hp_event)
    if (ev) cudaEventDestroy(ev);
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
      if (v < 0 || v > (int64_t{1} << 24)) return GEMM_ERR_INVALID_ARG;
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
    case GEMM_OPT_TF32_TRANSPOSE:
      if (v < 0 || v > 1) return GEMM_ERR_INVALID_ARG;
      h->tf32_transpose = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_STAGE_K:
      if (v < 0 || v > 2) return GEMM_ERR_INVALID_ARG;
      h->stage_k = static_cast<int>(v);
      return GEMM_OK;
    case GEMM_OPT_TILE_ROWS:
      if (v != 0 && (v < 64 || v > kTcBlockM || v % 8)) return GEMM_ERR_INVALID_ARG;
      h->tile_rows = static_cast<int>(v);
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

GEMM_API gemm_status_t gemm_set_kernel_events(gemm_handle_t h, void *start_event,
                                              void *end_event) {
  if (!h || (start_event == nullptr) != (end_event == nullptr)) return GEMM_ERR_INVALID_ARG;
  h->kernel_events[0] = static_cast<cudaEvent_t>(start_event);
  h->kernel_events[1] = static_cast<cudaEvent_t>(end_event);
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
