// host_path.cu -- gemm_run_host: the product of operands in host memory, with the copies
// to and from the device pipelined against the product on the handle's own streams.
#include "api_internal.h"

using namespace gemm_gb300;
using namespace gemm_gb300::api;

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
  // (after a failure part of them exist: those are kept, the rest created on the next call)
  for (cudaStream_t &st : h->hp_stream)
    if (!st && cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess) {
      st = nullptr;
      return cuda_fail(cudaGetLastError(), "host pipeline streams");
    }
  for (cudaEvent_t &ev : h->hp_event)
    if (!ev && cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
      ev = nullptr;
      return cuda_fail(cudaGetLastError(), "host pipeline events");
    }
  h->hp_ready = true;
  return GEMM_OK;
}

}  // namespace

extern "C" {

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
    st = execute(h, P, pl, s_mm, false);
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

}  // extern "C"
