// fma_kernel.cu -- exact-fp32 tile kernel, operand staging (copy or transpose) and zero fill.
//
// The FMA kernel is the blocked matrix multiply of "Chapter 13: The Blocked Matmul
// Kernel", section 13.1, Worked Example 13.1.1, done with fp32 fused multiply-adds:
// one CTA per BM x BN output tile on a 2D grid (ceil(N/BN), ceil(M/BM)), a K-loop of
// ceil(K/BK) chunks, an fp32 accumulator initialised once before the loop, loads masked
// by rows < M, k < K and cols < N with zeros outside (section 13.2's three masks), and a
// store masked by rows < M and cols < N. It serves the exact-fp32 mode ("Triton matmul",
// the "Precision" section: tf32 is not exact) and, with 4 x 4 x 4 tiles, the pages' own
// 8 x 8 x 8 example (grid 2 x 2, two K-iterations per tile). With an fp16 accumulator
// (section 13.3, Worked Example 13.3.1) each K-chunk's dot product is summed in fp32, then
// rounded to fp16 and added to the fp16 running total, itself rounded to fp16 after every
// chunk; the chunk is a multiple of BK, so with BK = 8 it can be the pages' own BLOCK_K.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace gemm_gb300 {
namespace {

template <typename T>
__device__ __forceinline__ float load_as_float(const void *base, int64_t idx) {
  return static_cast<float>(reinterpret_cast<const T *>(base)[idx]);
}
template <>
__device__ __forceinline__ float load_as_float<__half>(const void *base, int64_t idx) {
  return __half2float(reinterpret_cast<const __half *>(base)[idx]);
}
template <>
__device__ __forceinline__ float load_as_float<__nv_bfloat16>(const void *base, int64_t idx) {
  return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(base)[idx]);
}

__device__ __forceinline__ void store_out(void *C, int64_t idx, int out_dtype, float v) {
  if (out_dtype == GEMM_F32)
    reinterpret_cast<float *>(C)[idx] = v;
  else if (out_dtype == GEMM_BF16)
    reinterpret_cast<__nv_bfloat16 *>(C)[idx] = __float2bfloat16_rn(v);
  else
    reinterpret_cast<__half *>(C)[idx] = __float2half_rn(v);
}

// Row (or column) of the tile owned by thread coordinate t for its i-th register. With
// 8 registers the thread's rows are split into two groups of 4, half a tile apart, so
// that the shared-memory reads of a warp fall into distinct banks.
template <int T, int BLK>
__device__ __forceinline__ int owned(int t, int i) {
  if (T >= 8) return i < T / 2 ? t * (T / 2) + i : BLK / 2 + t * (T / 2) + (i - T / 2);
  return t * T + i;
}

// fp16(acc + fp16(partial)) for acc holding an fp16 value: the fp32 sum of two fp16 values
// rounded to fp16 equals their correctly rounded fp16 sum (fp32 carries 24 >= 2 * 11 + 2
// significand bits, so the double rounding is innocuous).
__device__ __forceinline__ float f16_accumulate(float acc, float partial) {
  const float h = __half2float(__float2half_rn(partial));
  return __half2float(__float2half_rn(acc + h));
}

// The K-loop keeps two chunks of A and B in shared memory: while the threads multiply one,
// the next chunk's elements are already on their way from global memory into registers and
// go to the other buffer after the products, so a chunk's load latency overlaps the
// previous chunk's arithmetic and each chunk needs one barrier.
template <int BM, int BN, int BK, int TM, int TN, typename InT, bool F16ACC>
__global__ void __launch_bounds__((BM / TM) * (BN / TN),
                                  (BM / TM) * (BN / TN) >= 256 && !F16ACC ? 2 : 1)
    fma_gemm_kernel(const FmaParams p) {
  constexpr int TX = BN / TN, TY = BM / TM, NT = TX * TY;
  constexpr int LA = (BM * BK + NT - 1) / NT, LB = (BK * BN + NT - 1) / NT;  // loads a thread
  __shared__ float As[2][BK][BM];
  __shared__ float Bs[2][BK][BN];
  const int tid = threadIdx.x;
  const int tx = tid % TX, ty = tid / TX;
  const int64_t m0 = static_cast<int64_t>(blockIdx.y) * BM;
  const int64_t n0 = static_cast<int64_t>(blockIdx.x) * BN;

  float acc[TM][TN];   // fp32 accumulator, or the chunk's partial dot (fp16 accumulator)
  float hacc[F16ACC ? TM : 1][F16ACC ? TN : 1];  // fp16 running total (fp16 accumulator)
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;  // initialised once, before the K-loop
  if (F16ACC) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) hacc[F16ACC ? i : 0][F16ACC ? j : 0] = 0.0f;
  }

  // Element e of a chunk, walking each operand's contiguous axis fastest; zero outside
  // rows < M, k < K, cols < N.
  float ra[LA], rb[LB];
  auto load_chunk = [&](int64_t k0) {
#pragma unroll
    for (int l = 0; l < LA; ++l) {
      const int e = tid + l * NT;
      float v = 0.0f;
      if (e < BM * BK) {
        const int r = p.a_col ? e % BM : e / BK;
        const int kk = p.a_col ? e / BM : e % BK;
        const int64_t i = m0 + r, k = k0 + kk;
        if (i < p.M && k < p.K)
          v = load_as_float<InT>(p.A, p.a_col ? k * p.lda + i : i * p.lda + k);
      }
      ra[l] = v;
    }
#pragma unroll
    for (int l = 0; l < LB; ++l) {
      const int e = tid + l * NT;
      float v = 0.0f;
      if (e < BK * BN) {
        const int c = p.b_col ? e / BK : e % BN;
        const int kk = p.b_col ? e % BK : e / BN;
        const int64_t j = n0 + c, k = k0 + kk;
        if (j < p.N && k < p.K)
          v = load_as_float<InT>(p.B, p.b_col ? j * p.ldb + k : k * p.ldb + j);
      }
      rb[l] = v;
    }
  };
  auto store_chunk = [&](int buf) {
#pragma unroll
    for (int l = 0; l < LA; ++l) {
      const int e = tid + l * NT;
      if (e < BM * BK) As[buf][p.a_col ? e / BM : e % BK][p.a_col ? e % BM : e / BK] = ra[l];
    }
#pragma unroll
    for (int l = 0; l < LB; ++l) {
      const int e = tid + l * NT;
      if (e < BK * BN) Bs[buf][p.b_col ? e % BK : e / BN][p.b_col ? e / BK : e % BN] = rb[l];
    }
  };

  load_chunk(0);
  store_chunk(0);
  __syncthreads();
  int buf = 0;
  for (int64_t k0 = 0; k0 < p.K; k0 += BK) {
    const bool more = k0 + BK < p.K;
    if (more) load_chunk(k0 + BK);  // in flight during the products below
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[TM], b[TN];
#pragma unroll
      for (int i = 0; i < TM; ++i) a[i] = As[buf][kk][owned<TM, BM>(ty, i)];
#pragma unroll
      for (int j = 0; j < TN; ++j) b[j] = Bs[buf][kk][owned<TN, BN>(tx, j)];
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    // the other buffer was last read before the previous barrier
    if (more) store_chunk(buf ^ 1);
    __syncthreads();
    buf ^= 1;
    if (F16ACC && ((k0 + BK) % p.acc_chunk == 0 || k0 + BK >= p.K)) {  // chunk done
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) {
          float &h = hacc[F16ACC ? i : 0][F16ACC ? j : 0];
          h = f16_accumulate(h, acc[i][j]);
          acc[i][j] = 0.0f;
        }
    }
  }
  if (F16ACC) {
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = hacc[F16ACC ? i : 0][F16ACC ? j : 0];
  }

#pragma unroll
  for (int i = 0; i < TM; ++i) {
    const int64_t row = m0 + owned<TM, BM>(ty, i);
    if (row >= p.M) continue;
#pragma unroll
    for (int j = 0; j < TN; ++j) {
      const int64_t col = n0 + owned<TN, BN>(tx, j);
      if (col < p.N) store_out(p.C, row * p.ldc + col, p.out_dtype, acc[i][j]);
    }
  }
}

template <int BM, int BN, int BK, int TM, int TN>
cudaError_t fma_launch_tile(const FmaParams &p, cudaStream_t s) {
  const dim3 grid(static_cast<unsigned>((p.N + BN - 1) / BN),
                  static_cast<unsigned>((p.M + BM - 1) / BM));
  const dim3 block((BM / TM) * (BN / TN));
  if (p.acc_chunk > 0) {
    if (p.in_dtype != GEMM_F16 || p.acc_chunk % BK) return cudaErrorInvalidValue;
    fma_gemm_kernel<BM, BN, BK, TM, TN, __half, true><<<grid, block, 0, s>>>(p);
  } else if (p.in_dtype == GEMM_F32) {
    fma_gemm_kernel<BM, BN, BK, TM, TN, float, false><<<grid, block, 0, s>>>(p);
  } else if (p.in_dtype == GEMM_F16) {
    fma_gemm_kernel<BM, BN, BK, TM, TN, __half, false><<<grid, block, 0, s>>>(p);
  } else {
    fma_gemm_kernel<BM, BN, BK, TM, TN, __nv_bfloat16, false><<<grid, block, 0, s>>>(p);
  }
  return cudaGetLastError();
}

template <typename T>
__global__ void repack_kernel(const T *__restrict__ src, int64_t ld_src, T *__restrict__ dst,
                              int64_t ld_dst, int64_t outer, int64_t inner) {
  for (int64_t o = blockIdx.y; o < outer; o += gridDim.y)
    for (int64_t x = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; x < inner;
         x += static_cast<int64_t>(gridDim.x) * blockDim.x)
      dst[o * ld_dst + x] = src[o * ld_src + x];
}

// dst[x * ld_dst + o] = src[o * ld_src + x]: `outer` source lines of `inner` elements
// become `inner` lines of `outer` elements. A CTA moves a strip of 32 source lines by 512
// contiguous bytes through shared memory: each warp reads 128-byte pieces of one source
// line (consecutive pieces back to back, so every DRAM page is read in long runs) and
// writes 128-byte pieces of one destination line; the odd row pitch of the staging tile
// keeps both directions free of bank conflicts.
template <typename T>
__global__ void __launch_bounds__(256) transpose_kernel(const T *__restrict__ src, int64_t ld_src,
                                                        T *__restrict__ dst, int64_t ld_dst,
                                                        int64_t outer, int64_t inner) {
  constexpr int S = 512 / (32 * sizeof(T));  // 32-element pieces per strip line
  __shared__ T tile[32][32 * S + 1];
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int64_t o0 = static_cast<int64_t>(blockIdx.y) * 32; o0 < outer;
       o0 += static_cast<int64_t>(gridDim.y) * 32) {
    for (int64_t x0 = static_cast<int64_t>(blockIdx.x) * 32 * S; x0 < inner;
         x0 += static_cast<int64_t>(gridDim.x) * 32 * S) {
      for (int j = ty; j < 32; j += blockDim.y) {
        const int64_t o = o0 + j;
#pragma unroll
        for (int s = 0; s < S; ++s) {
          const int64_t x = x0 + s * 32 + tx;
          if (o < outer && x < inner) tile[j][s * 32 + tx] = src[o * ld_src + x];
        }
      }
      __syncthreads();
#pragma unroll
      for (int s = 0; s < S; ++s) {
        for (int j = ty; j < 32; j += blockDim.y) {
          const int64_t x = x0 + s * 32 + j, o = o0 + tx;
          if (x < inner && o < outer) dst[x * ld_dst + o] = tile[tx][s * 32 + j];
        }
      }
      __syncthreads();
    }
  }
}

template <typename T>
__global__ void zero_fill_kernel(T *C, int64_t ldc, int64_t M, int64_t N) {
  for (int64_t i = blockIdx.y; i < M; i += gridDim.y)
    for (int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; j < N;
         j += static_cast<int64_t>(gridDim.x) * blockDim.x)
      C[i * ldc + j] = T(0);
}

dim3 grid_2d(int64_t outer, int64_t inner, int threads) {
  const int64_t gx = (inner + threads - 1) / threads;
  return dim3(static_cast<unsigned>(gx < 64 ? (gx < 1 ? 1 : gx) : 64),
              static_cast<unsigned>(outer < 65535 ? (outer < 1 ? 1 : outer) : 65535));
}

}  // namespace

// Tile kinds: 4 (the pages' 4 x 4 x 4 tiles), 8 (128 x 128 tiles, 8-long K-chunks: the
// fp16 accumulator, whose chunks are multiples of 8) and 128 (128 x 128 tiles, 16-long
// K-chunks: half the chunks, and barriers, over a long K).
void fma_tile_shape(int tile, int *bm, int *bn, int *bk) {
  if (tile == 4) {
    *bm = 4, *bn = 4, *bk = 4;
  } else {
    *bm = 128, *bn = 128, *bk = tile == 8 ? 8 : 16;
  }
}

cudaError_t fma_launch(const FmaParams &p, int tile, cudaStream_t s) {
  if (tile == 4) return fma_launch_tile<4, 4, 4, 1, 1>(p, s);
  if (tile == 8) return fma_launch_tile<128, 128, 8, 8, 8>(p, s);
  return fma_launch_tile<128, 128, 16, 8, 8>(p, s);
}

cudaError_t repack_launch(const void *src, int64_t ld_src, void *dst, int64_t ld_dst,
                          int64_t outer, int64_t inner, int esize, cudaStream_t s) {
  const int threads = 256;
  const dim3 grid = grid_2d(outer, inner, threads);
  if (esize == 2)
    repack_kernel<uint16_t><<<grid, threads, 0, s>>>(static_cast<const uint16_t *>(src), ld_src,
                                                     static_cast<uint16_t *>(dst), ld_dst, outer,
                                                     inner);
  else
    repack_kernel<uint32_t><<<grid, threads, 0, s>>>(static_cast<const uint32_t *>(src), ld_src,
                                                     static_cast<uint32_t *>(dst), ld_dst, outer,
                                                     inner);
  return cudaGetLastError();
}

cudaError_t transpose_launch(const void *src, int64_t ld_src, void *dst, int64_t ld_dst,
                             int64_t outer, int64_t inner, int esize, cudaStream_t s) {
  const dim3 block(32, 8);
  const int64_t strip = 512 / esize;  // source elements per strip line
  const int64_t gx = (inner + strip - 1) / strip, gy = (outer + 31) / 32;
  const dim3 grid(static_cast<unsigned>(gx < 4096 ? (gx < 1 ? 1 : gx) : 4096),
                  static_cast<unsigned>(gy < 4096 ? (gy < 1 ? 1 : gy) : 4096));
  if (esize == 2)
    transpose_kernel<uint16_t><<<grid, block, 0, s>>>(static_cast<const uint16_t *>(src), ld_src,
                                                      static_cast<uint16_t *>(dst), ld_dst, outer,
                                                      inner);
  else
    transpose_kernel<uint32_t><<<grid, block, 0, s>>>(static_cast<const uint32_t *>(src), ld_src,
                                                      static_cast<uint32_t *>(dst), ld_dst, outer,
                                                      inner);
  return cudaGetLastError();
}

cudaError_t zero_fill_launch(void *C, int64_t ldc, int64_t M, int64_t N, int out_dtype,
                             cudaStream_t s) {
  const int threads = 256;
  const dim3 grid = grid_2d(M, N, threads);
  if (out_dtype == GEMM_F32)
    zero_fill_kernel<uint32_t><<<grid, threads, 0, s>>>(static_cast<uint32_t *>(C), ldc, M, N);
  else
    zero_fill_kernel<uint16_t><<<grid, threads, 0, s>>>(static_cast<uint16_t *>(C), ldc, M, N);
  return cudaGetLastError();
}

}  // namespace gemm_gb300
