// split_kernel.cu -- operand staging for the exact-fp32 mode on tensor cores.
//
// Exact fp32 ("Triton matmul", "Precision": tf32 keeps only 10 mantissa bits, so fp32
// inputs need an explicit choice) is run on the tf32 tensor cores by splitting every fp32
// value x into two tf32 values, x = hi + lo + r with hi = tf32(x) and lo = tf32(x - hi),
// both rounded to nearest; |r| <= 2^-22 |x|. The product a*b is then
// hi_a*hi_b + hi_a*lo_b + lo_a*hi_b up to about 2^-21 |a*b| (the dropped lo_a*lo_b and the
// r terms), and the three partial products are one tf32 GEMM over a K-concatenated pair of
// operands:
//
//     A' = [hi(A) | hi(A) | lo(A)]   (M x 3K),   B' = [hi(B) ; lo(B) ; hi(B)]   (3K x N),
//
// so C = A' B' accumulates in the fp32 TMEM accumulator like any other product. This
// kernel writes A' or B' in K-major form (K contiguous, 3K + padding per row), transposing
// operands whose storage is not K-contiguous.
#include "internal.h"

namespace gemm_gb300 {
namespace {

__device__ __forceinline__ float tf32_rn(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// Writes the three segments of row r, column k of the split operand.
__device__ __forceinline__ void put3(float *dst, int64_t ldd, int64_t K, int64_t r, int64_t k,
                                     float x, bool is_b) {
  const float hi = tf32_rn(x);
  const float lo = tf32_rn(x - hi);
  float *row = dst + r * ldd + k;
  row[0] = hi;                 // segment 0: hi for A and for B
  row[K] = is_b ? lo : hi;     // segment 1: A's hi against B's lo
  row[2 * K] = is_b ? hi : lo; // segment 2: A's lo against B's hi
}

// Logical operand X[r][k] (R rows, K columns of the contraction). When k_contig, X[r][k]
// is src[r * lds + k]; otherwise src[k * lds + r] and the tile goes through shared memory
// so that both the reads and the writes are coalesced.
template <bool K_CONTIG>
__global__ void split3_kernel(const float *__restrict__ src, int64_t lds, float *__restrict__ dst,
                              int64_t ldd, int64_t R, int64_t K, bool is_b) {
  __shared__ float tile[32][33];
  for (int64_t r0 = static_cast<int64_t>(blockIdx.y) * 32; r0 < R;
       r0 += static_cast<int64_t>(gridDim.y) * 32) {
    for (int64_t k0 = static_cast<int64_t>(blockIdx.x) * 32; k0 < K;
         k0 += static_cast<int64_t>(gridDim.x) * 32) {
      if (K_CONTIG) {
        for (int j = threadIdx.y; j < 32; j += blockDim.y) {
          const int64_t r = r0 + j, k = k0 + threadIdx.x;
          if (r < R && k < K) put3(dst, ldd, K, r, k, src[r * lds + k], is_b);
        }
      } else {
        for (int j = threadIdx.y; j < 32; j += blockDim.y) {
          const int64_t k = k0 + j, r = r0 + threadIdx.x;
          if (k < K && r < R) tile[j][threadIdx.x] = src[k * lds + r];
        }
        __syncthreads();
        for (int j = threadIdx.y; j < 32; j += blockDim.y) {
          const int64_t r = r0 + j, k = k0 + threadIdx.x;
          if (r < R && k < K) put3(dst, ldd, K, r, k, tile[threadIdx.x][j], is_b);
        }
        __syncthreads();
      }
    }
  }
}

}  // namespace

cudaError_t split3_launch(const float *src, int64_t lds, bool k_contig, float *dst, int64_t ldd,
                          int64_t R, int64_t K, bool is_b, cudaStream_t s) {
  const dim3 block(32, 8);
  const int64_t gx = (K + 31) / 32, gy = (R + 31) / 32;
  const dim3 grid(static_cast<unsigned>(gx < 4096 ? (gx < 1 ? 1 : gx) : 4096),
                  static_cast<unsigned>(gy < 4096 ? (gy < 1 ? 1 : gy) : 4096));
  if (k_contig)
    split3_kernel<true><<<grid, block, 0, s>>>(src, lds, dst, ldd, R, K, is_b);
  else
    split3_kernel<false><<<grid, block, 0, s>>>(src, lds, dst, ldd, R, K, is_b);
  return cudaGetLastError();
}

}  // namespace gemm_gb300
