// strided.cu -- gemm_run_strided / gemm_plan_strided: any 2-D views of A, B and C.
#include "api_internal.h"

using namespace gemm_gb300;
using namespace gemm_gb300::api;

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

extern "C" {

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

}  // extern "C"
