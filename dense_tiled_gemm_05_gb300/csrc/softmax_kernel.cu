// softmax_kernel.cu -- row softmax, the second workload of the pages ("Triton from zero,
// Lesson 4: Block Pointers", homework 4): per row of an M x N matrix,
//
//     y_j = exp(x_j - m) / l,   m = max_k x_k,   l = sum_k exp(x_k - m),
//
// where the tile's columns past N are set to -inf before the max, so that they add
// exp(-inf) = 0 to the sum. The homework's kernel holds a whole row in one tile; here one
// CTA owns a row: its threads load the row into registers once (16-byte vector loads when
// the row is aligned; the columns past N take -inf), reduce the max and then the sum with
// warp shuffles and a shared-memory step, and write the row once -- one read and one write
// of HBM per element, the bound for this operation. Rows too long for registers (over
// 32 values per thread at 1024 threads) stream twice: a first pass keeps a running maximum
// and a sum rescaled whenever the maximum grows, a second pass writes the outputs. All
// arithmetic is fp32.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"

namespace gemm_gb300 {
namespace {

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half v) { return __half2float(v); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ T from_f32(float v);
template <>
__device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ __half from_f32<__half>(float v) { return __float2half_rn(v); }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Block-wide reduction of one float (max or sum) over T threads; every thread gets it.
template <int T, bool MAX>
__device__ __forceinline__ float block_reduce(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = MAX ? fmaxf(v, w) : v + w;
  }
  if (T == 32) return v;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  __syncthreads();  // red[] is reused by consecutive reductions
  if (lane == 0) red[warp] = v;
  __syncthreads();
  v = lane < T / 32 ? red[lane] : (MAX ? -INFINITY : 0.0f);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float w = __shfl_xor_sync(0xffffffffu, v, o);
    v = MAX ? fmaxf(v, w) : v + w;
  }
  return v;
}

// One CTA of T threads per row; each thread holds CH chunks of VEC consecutive columns:
// chunk c of thread t covers columns ((c * T + t) * VEC ..).
// (1024 / T CTAs per SM: at most 64 registers a thread, so that 1024 threads -- several
// rows -- stay resident on every SM)
template <typename TI, typename TO, int T, int CH, bool VECTOR>
__global__ void __launch_bounds__(T, 1024 / T) softmax_rows_kernel(const TI *__restrict__ X, int64_t ldx,
                                                         TO *__restrict__ Y, int64_t ldy,
                                                         int64_t M, int64_t N) {
  constexpr int VEC = 16 / sizeof(TI);
  __shared__ float red[32];
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const TI *x = X + row * ldx;
    float v[CH][VEC];
    float m = -INFINITY;
    bool has_nan = false;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int64_t j0 = (static_cast<int64_t>(c) * T + threadIdx.x) * VEC;
      if (VECTOR && j0 + VEC <= N) {
        const uint4 raw = *reinterpret_cast<const uint4 *>(x + j0);
        const TI *e = reinterpret_cast<const TI *>(&raw);
#pragma unroll
        for (int i = 0; i < VEC; ++i) v[c][i] = to_f32(e[i]);
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i) v[c][i] = j0 + i < N ? to_f32(x[j0 + i]) : -INFINITY;
      }
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        has_nan |= v[c][i] != v[c][i];
        m = fmaxf(m, v[c][i]);
      }
    }
    m = block_reduce<T, true>(m, red);
    // fmaxf drops NaN: a NaN anywhere in the row makes the whole row NaN, as in the formula
    if (__syncthreads_or(has_nan)) m = __int_as_float(0x7fffffff);
    float l = 0.0f;
#pragma unroll
    for (int c = 0; c < CH; ++c)
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        v[c][i] = expf(v[c][i] - m);  // -inf columns (padding) give exactly 0
        l += v[c][i];
      }
    l = block_reduce<T, false>(l, red);
    TO *y = Y + row * ldy;
#pragma unroll
    for (int c = 0; c < CH; ++c) {
      const int64_t j0 = (static_cast<int64_t>(c) * T + threadIdx.x) * VEC;
      if (VECTOR && j0 + VEC <= N && sizeof(TO) * VEC % 16 == 0) {
        TO out[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) out[i] = from_f32<TO>(v[c][i] / l);
        constexpr int W = sizeof(TO) * VEC / 16;  // 16-byte stores
#pragma unroll
        for (int w = 0; w < W; ++w)
          reinterpret_cast<uint4 *>(y + j0)[w] = reinterpret_cast<const uint4 *>(out)[w];
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i)
          if (j0 + i < N) y[j0 + i] = from_f32<TO>(v[c][i] / l);
      }
    }
  }
}

// VEC consecutive values of a row from column j0 (16-byte load when the row is aligned and
// the piece is whole); columns past N read as -inf.
template <typename TI, bool VECTOR>
__device__ __forceinline__ void load_piece(const TI *x, int64_t j0, int64_t N,
                                           float (&v)[16 / sizeof(TI)]) {
  constexpr int VEC = 16 / sizeof(TI);
  if (VECTOR && j0 + VEC <= N) {
    const uint4 raw = *reinterpret_cast<const uint4 *>(x + j0);
    const TI *e = reinterpret_cast<const TI *>(&raw);
#pragma unroll
    for (int i = 0; i < VEC; ++i) v[i] = to_f32(e[i]);
  } else {
#pragma unroll
    for (int i = 0; i < VEC; ++i) v[i] = j0 + i < N ? to_f32(x[j0 + i]) : -INFINITY;
  }
}

// Rows longer than the register kernel holds: two passes over the row (the second mostly
// from L2: the rows in flight fit in it). The first keeps, per thread, the maximum m of its
// values and l = sum exp(x - m), rescaling l whenever a piece raises m; the block then
// combines the (m, l) pairs. A NaN or +inf anywhere makes the row NaN (the formula's x - m
// is NaN there); a row of -inf only gives NaN through -inf - -inf. 512 threads, two CTAs
// (two rows) per SM.
template <typename TI, typename TO, bool VECTOR>
__global__ void __launch_bounds__(512, 2) softmax_rows_online_kernel(const TI *__restrict__ X,
                                                                     int64_t ldx,
                                                                     TO *__restrict__ Y,
                                                                     int64_t ldy, int64_t M,
                                                                     int64_t N) {
  constexpr int T = 512;
  constexpr int VEC = 16 / sizeof(TI);
  __shared__ float red[32];
  for (int64_t row = blockIdx.x; row < M; row += gridDim.x) {
    const TI *x = X + row * ldx;
    float m = -INFINITY, l = 0.0f;
    bool bad = false;
    for (int64_t j0 = static_cast<int64_t>(threadIdx.x) * VEC; j0 < N;
         j0 += static_cast<int64_t>(T) * VEC) {
      float v[VEC];
      load_piece<TI, VECTOR>(x, j0, N, v);
      float pm = -INFINITY;
#pragma unroll
      for (int i = 0; i < VEC; ++i) {
        bad |= v[i] != v[i] || v[i] == INFINITY;
        pm = fmaxf(pm, v[i]);
      }
      if (pm > m) {
        l *= expf(m - pm);  // rescale the sum to the new maximum (0 while m is -inf)
        m = pm;
      }
#pragma unroll
      for (int i = 0; i < VEC; ++i)
        if (v[i] != -INFINITY) l += expf(v[i] - m);
    }
    const float row_m = block_reduce<T, true>(m, red);
    const float lt = m == -INFINITY ? 0.0f : l * expf(m - row_m);
    const float row_l = block_reduce<T, false>(lt, red);
    const float mm = __syncthreads_or(bad) ? __int_as_float(0x7fffffff) : row_m;
    TO *y = Y + row * ldy;
    for (int64_t j0 = static_cast<int64_t>(threadIdx.x) * VEC; j0 < N;
         j0 += static_cast<int64_t>(T) * VEC) {
      float v[VEC];
      load_piece<TI, VECTOR>(x, j0, N, v);
      if (VECTOR && j0 + VEC <= N && sizeof(TO) * VEC % 16 == 0) {
        TO out[VEC];
#pragma unroll
        for (int i = 0; i < VEC; ++i) out[i] = from_f32<TO>(expf(v[i] - mm) / row_l);
#pragma unroll
        for (int w = 0; w < static_cast<int>(sizeof(TO) * VEC / 16); ++w)
          reinterpret_cast<uint4 *>(y + j0)[w] = reinterpret_cast<const uint4 *>(out)[w];
      } else {
#pragma unroll
        for (int i = 0; i < VEC; ++i)
          if (j0 + i < N) y[j0 + i] = from_f32<TO>(expf(v[i] - mm) / row_l);
      }
    }
  }
}

template <typename TI, typename TO, int T, int CH>
cudaError_t launch_rows(const void *X, int64_t ldx, void *Y, int64_t ldy, int64_t M, int64_t N,
                        bool vector, int grid, cudaStream_t s) {
  if (vector)
    softmax_rows_kernel<TI, TO, T, CH, true><<<grid, T, 0, s>>>(
        static_cast<const TI *>(X), ldx, static_cast<TO *>(Y), ldy, M, N);
  else
    softmax_rows_kernel<TI, TO, T, CH, false><<<grid, T, 0, s>>>(
        static_cast<const TI *>(X), ldx, static_cast<TO *>(Y), ldy, M, N);
  return cudaGetLastError();
}

template <typename TI, typename TO, int T>
cudaError_t launch_ch(const void *X, int64_t ldx, void *Y, int64_t ldy, int64_t M, int64_t N,
                      int64_t ch, bool vector, int grid, cudaStream_t s) {
  constexpr int MAX_CH = 32 / (16 / sizeof(TI));
  if (ch <= 1) return launch_rows<TI, TO, T, 1>(X, ldx, Y, ldy, M, N, vector, grid, s);
  if (ch <= 2) return launch_rows<TI, TO, T, 2>(X, ldx, Y, ldy, M, N, vector, grid, s);
  if (ch <= 4) return launch_rows<TI, TO, T, 4>(X, ldx, Y, ldy, M, N, vector, grid, s);
  return launch_rows<TI, TO, T, MAX_CH>(X, ldx, Y, ldy, M, N, vector, grid, s);
}

// Threads per row: the fewest (32 .. 1024, powers of two) that hold the row in registers
// at up to 32 values per thread. Few threads with many values each keep several rows per
// SM in flight: one row is loaded only while others reduce and store (bf16/fp32 rows of
// 8192 take 256 threads, four CTAs per SM).
template <typename TI, typename TO>
cudaError_t dispatch(const void *X, int64_t ldx, void *Y, int64_t ldy, int64_t M, int64_t N,
                     bool vector, int sm_count, cudaStream_t s) {
  constexpr int VEC = 16 / sizeof(TI);
  constexpr int MAX_CH = 32 / VEC;  // at most 32 fp32 values per thread
  const int64_t chunks = (N + VEC - 1) / VEC;
  const int64_t rows_cap = static_cast<int64_t>(sm_count > 0 ? sm_count : 1) * 64;
  const int grid = static_cast<int>(M < rows_cap ? M : rows_cap);
  if (chunks > 1024 * MAX_CH) {
    if (vector)
      softmax_rows_online_kernel<TI, TO, true><<<grid, 512, 0, s>>>(
          static_cast<const TI *>(X), ldx, static_cast<TO *>(Y), ldy, M, N);
    else
      softmax_rows_online_kernel<TI, TO, false><<<grid, 512, 0, s>>>(
          static_cast<const TI *>(X), ldx, static_cast<TO *>(Y), ldy, M, N);
    return cudaGetLastError();
  }
#define SOFTMAX_TRY(T_)                                                                        \
  if (chunks <= static_cast<int64_t>(T_) * MAX_CH)                                             \
    return launch_ch<TI, TO, T_>(X, ldx, Y, ldy, M, N, (chunks + T_ - 1) / T_, vector, grid, s);
  SOFTMAX_TRY(32)
  SOFTMAX_TRY(64)
  SOFTMAX_TRY(128)
  SOFTMAX_TRY(256)
  SOFTMAX_TRY(512)
#undef SOFTMAX_TRY
  return launch_ch<TI, TO, 1024>(X, ldx, Y, ldy, M, N, (chunks + 1023) / 1024, vector, grid, s);
}

template <typename TI>
cudaError_t dispatch_out(const void *X, int64_t ldx, void *Y, int64_t ldy, int64_t M, int64_t N,
                         int out_dtype, bool vector, int sm_count, cudaStream_t s) {
  if (out_dtype == GEMM_F32) return dispatch<TI, float>(X, ldx, Y, ldy, M, N, vector, sm_count, s);
  if (out_dtype == GEMM_F16) return dispatch<TI, __half>(X, ldx, Y, ldy, M, N, vector, sm_count, s);
  return dispatch<TI, __nv_bfloat16>(X, ldx, Y, ldy, M, N, vector, sm_count, s);
}

}  // namespace

cudaError_t softmax_rows_launch(const void *X, int64_t ldx, int in_dtype, void *Y, int64_t ldy,
                                int out_dtype, int64_t M, int64_t N, int sm_count,
                                cudaStream_t s) {
  if (M <= 0 || N <= 0) return cudaSuccess;
  const int ies = in_dtype == GEMM_F32 ? 4 : 2, oes = out_dtype == GEMM_F32 ? 4 : 2;
  // 16-byte vector loads (and stores) need every row to start on a 16-byte boundary
  const bool vector = reinterpret_cast<uintptr_t>(X) % 16 == 0 && (ldx * ies) % 16 == 0 &&
                      reinterpret_cast<uintptr_t>(Y) % 16 == 0 && (ldy * oes) % 16 == 0;
  if (in_dtype == GEMM_F32)
    return dispatch_out<float>(X, ldx, Y, ldy, M, N, out_dtype, vector, sm_count, s);
  if (in_dtype == GEMM_F16)
    return dispatch_out<__half>(X, ldx, Y, ldy, M, N, out_dtype, vector, sm_count, s);
  return dispatch_out<__nv_bfloat16>(X, ldx, Y, ldy, M, N, out_dtype, vector, sm_count, s);
}

}  // namespace gemm_gb300
