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

// The same operand stored the other way, X[r][k] = src[k * lds + r]: a CTA moves a tile
// of 32 k by 128 r through shared memory. Reads are 16-byte loads, eight lanes covering
// 128 contiguous bytes of one k-line; writes are 16-byte stores, eight lanes covering the
// 128 bytes of hi (and of lo) of one output row. In shared memory element (r, k) sits at
// r * 32 + (k ^ 4 * ((r / 4) % 8)): the XOR moves whole 4-float groups, so a row's four
// consecutive k stay one 16-byte word, and both the scalar stores of the load phase and
// the 16-byte loads of the write phase hit 32 different banks.
__global__ void __launch_bounds__(256) split2_cols_kernel(const float *__restrict__ src,
                                                          int64_t lds, float *__restrict__ dst,
                                                          int64_t ldd, int64_t R, int64_t K,
                                                          int64_t Kp, bool vec) {
  __shared__ __align__(16) float tile[128 * 32];
  const int lane = threadIdx.x % 32, w = threadIdx.x / 32;
  const int sub = lane / 8, q = lane % 8;  // 4 lines x 8 four-float groups per warp access
  auto at = [](int r, int k) { return r * 32 + (k ^ (4 * ((r >> 2) & 7))); };
  for (int64_t k0 = static_cast<int64_t>(blockIdx.y) * 32; k0 < Kp;
       k0 += static_cast<int64_t>(gridDim.y) * 32) {
    for (int64_t r0 = static_cast<int64_t>(blockIdx.x) * 128; r0 < R;
         r0 += static_cast<int64_t>(gridDim.x) * 128) {
      // load: warp w reads k-lines 4w..4w+3; pass i covers r 32i..32i+31
      const int kl = 4 * w + sub;
      const int64_t k = k0 + kl;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rl = 32 * i + 4 * q;
        const int64_t r = r0 + rl;
        float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
        if (k < K) {
          const float *p = src + k * lds + r;
          if (vec && r + 3 < R) {
            x = *reinterpret_cast<const float4 *>(p);
          } else {
            if (r < R) x.x = p[0];
            if (r + 1 < R) x.y = p[1];
            if (r + 2 < R) x.z = p[2];
            if (r + 3 < R) x.w = p[3];
          }
        }
        tile[at(rl + 0, kl)] = x.x;
        tile[at(rl + 1, kl)] = x.y;
        tile[at(rl + 2, kl)] = x.z;
        tile[at(rl + 3, kl)] = x.w;
      }
      __syncthreads();
      // write: pass i covers output rows 32i + 4w + sub, four k per lane
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int rl = 32 * i + 4 * w + sub;
        const int64_t r = r0 + rl;
        if (r < R) {
          const float4 x = *reinterpret_cast<const float4 *>(&tile[at(rl, 4 * q)]);
          const float4 hi = make_float4(tf32_rn(x.x), tf32_rn(x.y), tf32_rn(x.z), tf32_rn(x.w));
          const float4 lo = make_float4(tf32_rn(x.x - hi.x), tf32_rn(x.y - hi.y),
                                        tf32_rn(x.z - hi.z), tf32_rn(x.w - hi.w));
          float *row = dst + r * ldd + k0 + 4 * q;
          *reinterpret_cast<float4 *>(row) = hi;
          *reinterpret_cast<float4 *>(row + Kp) = lo;
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
    // 16-byte loads need a 16-byte aligned source and a pitch of whole 16-byte words
    const bool vec = reinterpret_cast<uintptr_t>(src) % 16 == 0 && lds % 4 == 0;
    const int64_t gx = (R + 127) / 128, gy = Kp / 32;
    const dim3 grid(static_cast<unsigned>(gx < 4096 ? gx : 4096),
                    static_cast<unsigned>(gy < 4096 ? gy : 4096));
    split2_cols_kernel<<<grid, 256, 0, s>>>(src, lds, dst, ldd, R, K, Kp, vec);
  }
  return cudaGetLastError();
}

}  // namespace gemm_gb300
