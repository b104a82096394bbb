// noalloc.cu -- gemm_run_noalloc, the allocation-free entry point (below).
#include <cstdio>
#include <mutex>

#include "api_internal.h"

using namespace gemm_gb300;
using namespace gemm_gb300::api;

// ---------------------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot call cudaMalloc at the point where they need a product: code that
// runs while a framework owns every device allocation (a plugin inside another runtime's
// memory pool), deployments that reserve all device memory up front and forbid growth,
// and host callbacks or real-time paths where a cudaMalloc (which may synchronise the
// device) is not allowed. gemm_run_noalloc serves them without a handle: the staging
// copies that misaligned operands and MN-major tf32 operands need, and the tf32 hi/lo
// split operands of exact fp32, go to a fixed, file-scope device array instead of a
// workspace that grows on demand.
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
      std::fprintf(stderr, "[gemm] gemm_run_noalloc: %s needs %lld bytes of scratch, limit %zu\n",
                   I.path == GEMM_PATH_TCGEN05_3XTF32 ? "exact fp32 (split operands)" : "staging",
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
  // Split-K keeps its partial tiles in a handle-owned workspace: plan whole tiles only.
  Options whole;
  whole.stream_k = 1;
  st = make_plan(P, whole, sms, &pl);
  if (st != GEMM_OK) return st;
  // Staged copies and the split hi/lo operands of exact fp32 alike must fit the array;
  // a problem that needs more is refused (execute_noalloc) before anything is launched.
  return execute_noalloc(scratch, device_status, P, pl, static_cast<cudaStream_t>(cuda_stream));
}
