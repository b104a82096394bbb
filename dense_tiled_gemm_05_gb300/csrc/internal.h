// internal.h -- declarations shared by the host runtime (gemm_api.cu) and the kernel
// translation units. Nothing here is part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gemm.h"

namespace gemm_gb300 {

// Debug flags carried into the tensor-core kernel (test hooks of
// GEMM_OPT_FAULT_STALL_PRODUCER): bit 0, every loader issues nothing; else bits 8.. give a
// number of stage fills after which a loader stops, that of CTA rank 1 of a pair when bit 1
// is set, of rank 0 otherwise (the single-CTA kernel's loader either way).
enum : int { kDebugStallProducer = 1, kDebugStallRank1 = 2, kDebugStallAfterShift = 8 };

// Stage fills after which this CTA's loader stops under the test hook (-1: never).
inline __host__ __device__ int stall_after_fills(int debug_flags, int rank) {
  const int n = debug_flags >> kDebugStallAfterShift;
  if (n <= 0) return -1;
  return ((debug_flags & kDebugStallRank1) ? 1 : 0) == rank ? n : -1;
}
// TcParams::l2_once bits: the operand is read by one tile column (A) or row (B) only.
enum : int { kL2OnceA = 1, kL2OnceB = 2 };
// TcParams::mn_3d bits: the MN-major operand's tensor map is 3D (one copy per stage).
enum : int { kMn3dA = 1, kMn3dB = 2 };

// Output tile of the tensor-core kernel: 128 rows (one TMEM lane per row).
constexpr int kTcBlockM = 128;

// Arguments of the persistent tensor-core kernel that are not tensor maps.
struct TcParams {
  int32_t M, N, K;
  int32_t tiles_m, tiles_n, k_blocks;
  int32_t group_m;     // tile rows per raster group
  uint32_t idesc;      // tcgen05 instruction descriptor
  int32_t out_dtype;   // gemm_dtype_t
  int32_t tma_store;   // 1: TMA-store epilogue; 0: masked st.global epilogue
  void *C;
  int64_t ldc;
  int *status;         // device status word
  uint64_t timeout_ns; // bounded-wait limit
  int32_t debug_flags;
  int32_t chunk_steps;    // chunked kernel: MMA instructions per TMEM partial sum
  int32_t cta_rows;       // rows of A each CTA loads per tile (CTA-pair kernel; <= 128)
  int32_t l2_once;        // kL2OnceA | kL2OnceB: operands loaded as first to evict from L2
  int32_t k_rotate;       // whole tile t starts at K-block (t * k_rotate) mod k_blocks (0: 0)
  int32_t split_kb;       // exact fp32: K-blocks per hi or lo part of the split operands
  int32_t mn_3d;          // kMn3dA | kMn3dB: MN-major operands loaded by one 3D copy a stage
  // split-K share of the last rounds (CTA-pair kernel; see sk_schedule.h)
  int32_t sk_dp_tiles;    // tiles done whole, round-robin (== tiles: no split)
  float *sk_partials;     // [worker][cta rank][128 rows][block_n] fp32
  int *sk_flags;          // [worker][cta rank][8]: one flag per epilogue warp (4 or 8 used)
  int *sk_epoch_word;     // [epoch, arrivals]: writers store epoch + 1 in their flags; the
                          // last CTA to finish advances the epoch (see tc_common.cuh)
};

// One tensor-core kernel variant: element size of A and B (2 = f16/bf16, 4 = fp32 as tf32),
// operand majorness, and the output tile width.
struct TcVariant {
  int esize;
  bool a_mn, b_mn;
  int block_n;
  bool pair;   // CTA pair (cta_group::2): 256-row tiles over two SMs
  bool exact;   // exact-fp32 kernel on split operands (CTA pairs, chunked fp32 sums)
  bool f16acc;  // fp16-accumulator kernel (CTA pairs, chunk dots rounded into fp16 sums)
  int kps = 1;  // CTA-pair kernel: 128-byte K-blocks per pipeline stage (1, or 2 for K-major
                // 16-bit operands)
};

int tc_stages(const TcVariant &v);
// tmP: the split-K partial tiles as a 2D fp32 tensor (CTA-pair kernel only).
cudaError_t tc_launch(const TcVariant &v, const CUtensorMap &tmA, const CUtensorMap &tmB,
                      const CUtensorMap &tmC, const CUtensorMap &tmP, const TcParams &p, int grid,
                      cudaStream_t s);
// CTA-pair kernel: grid counts CTAs (twice the clusters).
cudaError_t tc2_launch(const TcVariant &v, const CUtensorMap &tmA, const CUtensorMap &tmB,
                       const CUtensorMap &tmC, const CUtensorMap &tmP, const TcParams &p, int grid,
                       cudaStream_t s);
// Clusters of two CTAs of the pair kernel that fit on the current device at once.
int tc2_max_active_clusters();
// Chunked kernel (CTA pairs, 256 x 256 tiles, K-major operands, register accumulators):
// exact fp32 on split tf32 operands, or (f16acc) fp16 inputs with an fp16 accumulator.
// tmP: split-K partial tiles (exact mode), as for the CTA-pair kernel.
cudaError_t tc_chunk_launch(bool f16acc, const CUtensorMap &tmA, const CUtensorMap &tmB,
                            const CUtensorMap &tmC, const CUtensorMap &tmP, const TcParams &p,
                            int grid, cudaStream_t s);
int tc_chunk_max_active_clusters(bool f16acc);
// K-blocks of 32 split products the exact kernel accumulates in TMEM before adding the
// partial into its fp32 register sums. The tensor cores' accumulation keeps fewer bits
// than an IEEE fp32 add, and its error relative to sum |a b| is largest for short K, so
// short products use short chunks; long ones use up to 16 K-blocks (longer chunks only
// saved ~1 % more time on GB300).
inline int exact_chunk_kblocks(int64_t k_blocks) {
  const int64_t c = k_blocks / 24;
  return static_cast<int>(c < 1 ? 1 : c > 16 ? 16 : c);
}

// fp32 fused-multiply-add tile kernel (exact fp32 mode; any input dtype/layout).
struct FmaParams {
  int64_t M, N, K;
  const void *A;
  int64_t lda;
  const void *B;
  int64_t ldb;
  void *C;
  int64_t ldc;
  int32_t in_dtype, out_dtype;
  int32_t a_col, b_col;  // 1 = column-major operand
  int64_t acc_chunk;     // > 0: fp16 accumulator rounded every acc_chunk K (a multiple of BK)
};
// tile: 4 selects the 4x4x4 tiles of the pages' 8x8x8 example, anything else 128x128x8.
cudaError_t fma_launch(const FmaParams &p, int tile, cudaStream_t s);
void fma_tile_shape(int tile, int *bm, int *bn, int *bk);

// Copy a rows x cols operand (storage: `outer` lines of `inner` elements, leading dim
// ld_src) into dst with leading dim ld_dst. esize is 2 or 4 bytes.
cudaError_t repack_launch(const void *src, int64_t ld_src, void *dst, int64_t ld_dst,
                          int64_t outer, int64_t inner, int esize, cudaStream_t s);

// Transposing copy: source `outer` lines of `inner` elements (leading dim ld_src) become
// `inner` lines of `outer` elements in dst (leading dim ld_dst >= outer).
cudaError_t transpose_launch(const void *src, int64_t ld_src, void *dst, int64_t ld_dst,
                             int64_t outer, int64_t inner, int esize, cudaStream_t s);

// Exact-fp32 staging: writes the K-major operand [hi | lo] of R rows, each part K columns
// zero-padded to Kp (a multiple of 32; leading dim ldd >= 2 Kp, a multiple of 4; dst
// 16-byte aligned, else cudaErrorInvalidValue), from an fp32 operand X[r][k] stored
// K-contiguous (src[r*lds + k]) or not (src[k*lds + r]).
cudaError_t split2_launch(const float *src, int64_t lds, bool k_contig, float *dst, int64_t ldd,
                          int64_t R, int64_t K, int64_t Kp, cudaStream_t s);

// dst[i * d0 + j * d1] = src[i * s0 + j * s1] for i < n0, j < n1 (element strides; the
// source's may be 0). esize is 2 or 4 bytes.
cudaError_t strided_copy_launch(const void *src, int64_t s0, int64_t s1, void *dst, int64_t d0,
                                int64_t d1, int64_t n0, int64_t n1, int esize, cudaStream_t s);

// Row softmax y = exp(x - max) / sum(exp(x - max)) of an M x N row-major matrix (fp32
// arithmetic; any of the three dtypes in and out; X == Y with equal ld and dtype allowed).
cudaError_t softmax_rows_launch(const void *X, int64_t ldx, int in_dtype, void *Y, int64_t ldy,
                                int out_dtype, int64_t M, int64_t N, int sm_count,
                                cudaStream_t s);

// C[i, j] = 0 for i < M, j < N.
cudaError_t zero_fill_launch(void *C, int64_t ldc, int64_t M, int64_t N, int out_dtype,
                             cudaStream_t s);

}  // namespace gemm_gb300
