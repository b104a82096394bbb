// strided_kernel.cu -- copies between arbitrarily strided 2D views, for the six-stride
// interface ("Chapter 13: The Blocked Matmul Kernel", section 13.4: the host wrapper hands
// the kernel both strides of A, B and C, so any 2D view is an operand).
//
// dst[i * d0 + j * d1] = src[i * s0 + j * s1] for i < n0, j < n1. Each 32 x 32 tile goes
// through shared memory: it is read with consecutive lanes along the source's
// smaller-stride dimension and written with consecutive lanes along the destination's, so
// whichever of the two is contiguous is accessed in full 128-byte lines. Strides may be 0
// on the source (a broadcast view).
#include <cuda_runtime.h>

#include "internal.h"

namespace gemm_gb300 {
namespace {

template <typename T>
__global__ void strided_copy_kernel(const T *__restrict__ src, int64_t s0, int64_t s1,
                                    T *__restrict__ dst, int64_t d0, int64_t d1, int64_t n0,
                                    int64_t n1, bool src_fast1, bool dst_fast1) {
  __shared__ T tile[32][33];
  const int tx = threadIdx.x, ty = threadIdx.y;
  for (int64_t b0 = static_cast<int64_t>(blockIdx.y) * 32; b0 < n0;
       b0 += static_cast<int64_t>(gridDim.y) * 32) {
    for (int64_t b1 = static_cast<int64_t>(blockIdx.x) * 32; b1 < n1;
         b1 += static_cast<int64_t>(gridDim.x) * 32) {
      for (int j = ty; j < 32; j += blockDim.y) {
        const int r = src_fast1 ? j : tx, c = src_fast1 ? tx : j;
        if (b0 + r < n0 && b1 + c < n1) tile[r][c] = src[(b0 + r) * s0 + (b1 + c) * s1];
      }
      __syncthreads();
      for (int j = ty; j < 32; j += blockDim.y) {
        const int r = dst_fast1 ? j : tx, c = dst_fast1 ? tx : j;
        if (b0 + r < n0 && b1 + c < n1) dst[(b0 + r) * d0 + (b1 + c) * d1] = tile[r][c];
      }
      __syncthreads();
    }
  }
}

int64_t abs64(int64_t x) { return x < 0 ? -x : x; }

}  // namespace

cudaError_t strided_copy_launch(const void *src, int64_t s0, int64_t s1, void *dst, int64_t d0,
                                int64_t d1, int64_t n0, int64_t n1, int esize, cudaStream_t s) {
  if (n0 <= 0 || n1 <= 0) return cudaSuccess;
  // consecutive lanes along dimension 1 when its stride is the smaller one (or dim 0 has a
  // single element)
  const bool src_fast1 = n0 == 1 || abs64(s1) <= abs64(s0);
  const bool dst_fast1 = n0 == 1 || abs64(d1) <= abs64(d0);
  const dim3 block(32, 8);
  const int64_t gx = (n1 + 31) / 32, gy = (n0 + 31) / 32;
  const dim3 grid(static_cast<unsigned>(gx < 2048 ? gx : 2048),
                  static_cast<unsigned>(gy < 2048 ? gy : 2048));
  if (esize == 2)
    strided_copy_kernel<uint16_t><<<grid, block, 0, s>>>(
        static_cast<const uint16_t *>(src), s0, s1, static_cast<uint16_t *>(dst), d0, d1, n0,
        n1, src_fast1, dst_fast1);
  else
    strided_copy_kernel<uint32_t><<<grid, block, 0, s>>>(
        static_cast<const uint32_t *>(src), s0, s1, static_cast<uint32_t *>(dst), d0, d1, n0,
        n1, src_fast1, dst_fast1);
  return cudaGetLastError();
}

}  // namespace gemm_gb300
