// split_kernel.cu -- operand staging for the exact-fp32 mode on tensor cores.
//
// Exact fp32 ("Triton matmul", "Precision": tf32 keeps only 10 mantissa bits, so fp32
// inputs need an explicit choice) is run on the tf32 tensor cores by splitting every fp32
// value x into two tf32 values, x = hi + lo + r with hi = tf32(x) and lo = tf32(x - hi),
// both rounded to nearest; |r| <= 2^-22 |x|. The product a*b is then
// hi_a*hi_b + hi_a*lo_b + lo_a*hi_b up to about 2^-21 |a*b| (the dropped lo_a*lo_b and the
// r terms), three partial products over the same K.
//
// This kernel writes an operand's two parts side by side, K-major (K contiguous):
//
//     X2[r] = [hi(X[r][0..K)) 0..0 | lo(X[r][0..K)) 0..0]   (2 Kp columns),
//
// each part zero-padded from K to Kp, K rounded up to a whole 32-long K-block. The exact
// kernel reads the three products as 3 Kp / 32 K-blocks: K-block j of product q in {0, 1, 2}
// takes A's part (q == 2 ? lo : hi) and B's part (q == 1 ? lo : hi) at K-block j, so
// A' = [hi | hi | lo] and B' = [hi ; lo ; hi] are never written out. Operands whose storage
// is not K-contiguous are transposed on the way.
#include "internal.h"

namespace gemm_gb300 {
namespace {

__device__ __forceinline__ float tf32_rn(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return __uint_as_float(r);
}

// Writes both parts of row r, column k of the split operand (x = 0 in the padding).
__device__ __forceinline__ void put2(float *dst, int64_t ldd, int64_t Kp, int64_t r, int64_t k,
                                     float x) {
  const float hi = tf32_rn(x);
  float *row = dst + r * ldd + k;
  row[0] = hi;
  row[Kp] = tf32_rn(x - hi);
}

// Logical operand X[r][k] (R rows, K columns of the contraction), stored K-contiguous:
// X[r][k] = src[r * lds + k]. Each thread splits 4 consecutive k of one row: one 16-byte
// load and two 16-byte stores when the row is 16-byte aligned (scalar otherwise, at the
// row's ragged end, and in the zero padding up to Kp).
__global__ void __launch_bounds__(256) split2_rows_kernel(const float *__restrict__ src,
                                                          int64_t lds, float *__restrict__ dst,
                                                          int64_t ldd, int64_t R, int64_t K,
                                                          int64_t Kp, bool vec) {
  const int64_t kc = Kp / 4;  // 4-wide chunks per row (Kp is a multiple of 32)
  for (int64_t id = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; id < R * kc;
       id += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t r = id / kc, k = (id - r * kc) * 4;
    float4 *row = reinterpret_cast<float4 *>(dst + r * ldd + k);
    if (vec && k + 4 <= K) {
      const float4 x = *reinterpret_cast<const float4 *>(src + r * lds + k);
      const float4 hi = make_float4(tf32_rn(x.x), tf32_rn(x.y), tf32_rn(x.z), tf32_rn(x.w));
      row[0] = hi;
      row[Kp / 4] = make_float4(tf32_rn(x.x - hi.x), tf32_rn(x.y - hi.y), tf32_rn(x.z - hi.z),
                                tf32_rn(x.w - hi.w));
    } else if (k >= K) {
      row[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      row[Kp / 4] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      for (int64_t kk = k; kk < k + 4; ++kk) put2(dst, ldd, Kp, r, kk, kk < K ? src[r * lds + kk] : 0.f);
    }
  }
}

// The same operand stored the other way, X[r][k] = src[k * lds + r]: a CTA moves 32 lines
// of k by 512 contiguous bytes of r through shared memory (the strip transpose of the
// staging copy), so both the reads and the split writes are long contiguous runs.
__global__ void __launch_bounds__(256) split2_cols_kernel(const float *__restrict__ src,
                                                          int64_t lds, float *__restrict__ dst,
                                                          int64_t ldd, int64_t R, int64_t K,
                                                          int64_t Kp) {
  constexpr int S = 4;  // 32-float pieces per strip line (512 bytes)
  __shared__ float tile[32][32 * S + 1];
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int64_t k0 = static_cast<int64_t>(blockIdx.y) * 32; k0 < Kp;
       k0 += static_cast<int64_t>(gridDim.y) * 32) {
    for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * 32 * S; r0 < R;
         r0 += static_cast<int64_t>(gridDim.x) * 32 * S) {
      for (int j = ty; j < 32; j += blockDim.y) {
        const int64_t k = k0 + j;
#pragma unroll
        for (int s = 0; s < S; ++s) {
          const int64_t r = r0 + s * 32 + tx;
          if (r < R) tile[j][s * 32 + tx] = k < K ? src[k * lds + r] : 0.f;
        }
      }
      __syncthreads();
#pragma unroll
      for (int s = 0; s < S; ++s) {
        for (int j = ty; j < 32; j += blockDim.y) {
          const int64_t r = r0 + s * 32 + j, k = k0 + tx;
          if (r < R && k < Kp) put2(dst, ldd, Kp, r, k, tile[tx][s * 32 + j]);
        }
      }
      __syncthreads();
    }
  }
}

}  // namespace

cudaError_t split2_launch(const float *src, int64_t lds, bool k_contig, float *dst, int64_t ldd,
                          int64_t R, int64_t K, int64_t Kp, cudaStream_t s) {
  if (R <= 0 || K <= 0) return cudaSuccess;
  if (Kp % 32 != 0 || Kp < K || ldd < 2 * Kp || ldd % 4 != 0 ||
      reinterpret_cast<uintptr_t>(dst) % 16 != 0)
    return cudaErrorInvalidValue;
  if (k_contig) {
    // 16-byte loads need 16-byte aligned source rows (the destination always is)
    const bool vec = reinterpret_cast<uintptr_t>(src) % 16 == 0 && lds % 4 == 0;
    const int64_t chunks = R * (Kp / 4);
    const int64_t blocks = (chunks + 255) / 256;
    split2_rows_kernel<<<static_cast<unsigned>(blocks < 65536 ? blocks : 65536), 256, 0, s>>>(
        src, lds, dst, ldd, R, K, Kp, vec);
  } else {
    const dim3 block(32, 8);
    const int64_t gx = (R + 127) / 128, gy = Kp / 32;
    const dim3 grid(static_cast<unsigned>(gx < 4096 ? gx : 4096),
                    static_cast<unsigned>(gy < 4096 ? gy : 4096));
    split2_cols_kernel<<<grid, block, 0, s>>>(src, lds, dst, ldd, R, K, Kp);
  }
  return cudaGetLastError();
}

}  // namespace gemm_gb300
