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

// Logical operand X[r][k] (R rows, K columns of the contraction), stored K-contiguous:
// X[r][k] = src[r * lds + k]. Each thread splits 4 consecutive k of one row: one 16-byte
// load and three 16-byte stores when the row and the destination are 16-byte aligned
// (scalar otherwise, and at the row's ragged end).
__global__ void __launch_bounds__(256) split3_rows_kernel(const float *__restrict__ src,
                                                          int64_t lds, float *__restrict__ dst,
                                                          int64_t ldd, int64_t R, int64_t K,
                                                          bool is_b, bool vec) {
  const int64_t kc = (K + 3) / 4;  // 4-wide chunks per row
  for (int64_t id = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; id < R * kc;
       id += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = id / kc, k = (id - r * kc) * 4;
    if (vec && k + 4 <= K) {
      const float4 x = *reinterpret_cast<const float4 *>(src + r * lds + k);
      const float4 hi = make_float4(tf32_rn(x.x), tf32_rn(x.y), tf32_rn(x.z), tf32_rn(x.w));
      const float4 lo = make_float4(tf32_rn(x.x - hi.x), tf32_rn(x.y - hi.y), tf32_rn(x.z - hi.z),
                                    tf32_rn(x.w - hi.w));
      float4 *row = reinterpret_cast<float4 *>(dst + r * ldd + k);
      row[0] = hi;                             // segment 0: hi for A and for B
      row[K / 4] = is_b ? lo : hi;             // segment 1: A's hi against B's lo
      row[2 * (K / 4)] = is_b ? hi : lo;       // segment 2: A's lo against B's hi
    } else {
      for (int64_t kk = k; kk < k + 4 && kk < K; ++kk)
        put3(dst, ldd, K, r, kk, src[r * lds + kk], is_b);
    }
  }
}

// The same operand stored the other way, X[r][k] = src[k * lds + r]: a CTA moves 32 lines
// of k by 512 contiguous bytes of r through shared memory (the strip transpose of the
// staging copy), so both the reads and the split writes are long contiguous runs.
__global__ void __launch_bounds__(256) split3_cols_kernel(const float *__restrict__ src,
                                                          int64_t lds, float *__restrict__ dst,
                                                          int64_t ldd, int64_t R, int64_t K,
                                                          bool is_b) {
  constexpr int S = 4;  // 32-float pieces per strip line (512 bytes)
  __shared__ float tile[32][32 * S + 1];
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int64_t k0 = static_cast<int64_t>(blockIdx.y) * 32; k0 < K;
       k0 += static_cast<int64_t>(gridDim.y) * 32) {
    for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * 32 * S; r0 < R;
         r0 += static_cast<int64_t>(gridDim.x) * 32 * S) {
      for (int j = ty; j < 32; j += blockDim.y) {
        const int64_t k = k0 + j;
#pragma unroll
        for (int s = 0; s < S; ++s) {
          const int64_t r = r0 + s * 32 + tx;
          if (k < K && r < R) tile[j][s * 32 + tx] = src[k * lds + r];
        }
      }
      __syncthreads();
#pragma unroll
      for (int s = 0; s < S; ++s) {
        for (int j = ty; j < 32; j += blockDim.y) {
          const int64_t r = r0 + s * 32 + j, k = k0 + tx;
          if (r < R && k < K) put3(dst, ldd, K, r, k, tile[tx][s * 32 + j], is_b);
        }
      }
      __syncthreads();
    }
  }
}

}  // namespace

cudaError_t split3_launch(const float *src, int64_t lds, bool k_contig, float *dst, int64_t ldd,
                          int64_t R, int64_t K, bool is_b, cudaStream_t s) {
  if (R <= 0 || K <= 0) return cudaSuccess;
  if (k_contig) {
    // 16-byte accesses: the source rows, the destination rows and the segment offsets K
    // and 2K must all fall on 16-byte boundaries
    const bool vec = reinterpret_cast<uintptr_t>(src) % 16 == 0 && lds % 4 == 0 &&
                     reinterpret_cast<uintptr_t>(dst) % 16 == 0 && ldd % 4 == 0 && K % 4 == 0;
    const int64_t chunks = R * ((K + 3) / 4);
    const int64_t blocks = (chunks + 255) / 256;
    split3_rows_kernel<<<static_cast<unsigned>(blocks < 65536 ? blocks : 65536), 256, 0, s>>>(
        src, lds, dst, ldd, R, K, is_b, vec);
  } else {
    const dim3 block(32, 8);
    const int64_t gx = (R + 127) / 128, gy = (K + 31) / 32;
    const dim3 grid(static_cast<unsigned>(gx < 4096 ? gx : 4096),
                    static_cast<unsigned>(gy < 4096 ? gy : 4096));
    split3_cols_kernel<<<grid, block, 0, s>>>(src, lds, dst, ldd, R, K, is_b);
  }
  return cudaGetLastError();
}

}  // namespace gemm_gb300
