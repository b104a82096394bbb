// tc_kernel.cu -- the tensor-core blocked GEMM for sm_103a.
//
// The computation is the blocked matrix multiply of "Chapter 13: The Blocked Matmul
// Kernel", section 13.1: the output is a grid of BLOCK_M x BLOCK_N tiles, each tile walks
// ceil(K / BLOCK_K) K-chunks and adds every chunk's partial product into an fp32
// accumulator that is initialised once (the first MMA of a tile overwrites instead of
// accumulating). Section 13.2's three masks come from the TMA unit: a box that hangs off
// the tensor in M, N or K is zero-filled ("Triton from zero, Lesson 4: Block Pointers",
// section 3: zero padding is exact for a matmul), and the store is clipped to M x N.
// Section 13.3's single rounding happens in the epilogue: fp32 TMEM -> out dtype once.
//
// Structure (one CTA per SM, persistent over tiles):
//   warp 0        TMA producer: one elected lane streams A/B K-chunks into a STAGES-deep
//                 shared-memory ring (full/empty mbarriers);
//   warp 1        MMA issuer: one lane issues tcgen05.mma (M=128, N=BN, K=32 bytes) into a
//                 TMEM accumulator; the warp also owns the TMEM allocation;
//   warps 2..5    epilogue: tcgen05.ld -> convert -> swizzled staging -> TMA store (or a
//                 masked st.global when C is not TMA-legal).
// The accumulator is double-buffered in TMEM (2 x BN columns), so the epilogue of tile t
// overlaps the main loop of tile t+1. Tiles are visited in grouped raster order
// (GROUP_M tile-rows at a time) so that consecutive tiles on the machine share A and B
// panels in L2.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace gemm_gb300 {
namespace {

constexpr int kThreads = 192;
constexpr int kEpiWarps = 4;
constexpr int kRowBytes = 128;                   // one 128-byte swizzle row
constexpr int kStoreBufBytes = 32 * kRowBytes;   // one epilogue staging box: 32 rows x 128 B

template <int ESIZE, bool A_MN, bool B_MN, int BN>
struct Cfg {
  static constexpr int BM = kTcBlockM;
  static constexpr int BK = kRowBytes / ESIZE;         // K elements per stage (64 or 32)
  static constexpr int UMMA_K = 32 / ESIZE;            // K elements per tcgen05.mma
  static constexpr int K_STEPS = BK / UMMA_K;          // MMAs per stage
  static constexpr int PANEL = kRowBytes / ESIZE;      // M/N elements per 128-byte row (MN-major)
  static constexpr int PANEL_BYTES = BK * kRowBytes;   // MN-major panel: BK rows x 128 B
  static constexpr int A_BYTES = BM * BK * ESIZE;
  static constexpr int B_BYTES = BN * BK * ESIZE;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = BN >= 256 ? 4 : 6;
  static constexpr int EPI_OFFSET = STAGES * STAGE_BYTES;
  static constexpr int EPI_BYTES = kEpiWarps * 2 * kStoreBufBytes;
  static constexpr int BAR_OFFSET = EPI_OFFSET + EPI_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5;  // full[], empty[], tmem_full[2], tmem_empty[2], drain
  static constexpr int SMEM_BYTES = BAR_OFFSET + NUM_BARS * 8 + 16 + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(TMEM_COLS <= 512 && (TMEM_COLS & (TMEM_COLS - 1)) == 0, "TMEM allocation");
};

__device__ __forceinline__ void tile_coords(int tile, int tiles_m, int tiles_n, int group_m,
                                            int &pm, int &pn) {
  const int per_group = group_m * tiles_n;
  const int g = tile / per_group;
  const int first_m = g * group_m;
  const int gsize = min(tiles_m - first_m, group_m);
  const int r = tile - g * per_group;
  pm = first_m + r % gsize;
  pn = r / gsize;
}

// Time-bounded wait used only while tearing down after an abort: it ignores the abort
// flag (the point is to let in-flight copies and MMAs land) and records nothing.
__device__ __noinline__ void drain_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) return;
  }
}

__device__ __forceinline__ uint32_t pack2_bf16(uint32_t a, uint32_t b) {
  __nv_bfloat162 h = __floats2bfloat162_rn(__uint_as_float(a), __uint_as_float(b));
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ uint32_t pack2_f16(uint32_t a, uint32_t b) {
  __half2 h = __floats2half2_rn(__uint_as_float(a), __uint_as_float(b));
  return *reinterpret_cast<uint32_t *>(&h);
}

template <int OUT>
__device__ __forceinline__ uint32_t pack2(uint32_t a, uint32_t b) {
  return OUT == GEMM_BF16 ? pack2_bf16(a, b) : pack2_f16(a, b);
}

// Epilogue, TMA-store form: one 32-row slab of the tile per warp; each 128-byte-wide
// column block is converted, written to a 128B-swizzled staging box and stored by TMA
// (which clips rows >= M and columns >= N). Two staging boxes per warp alternate.
template <int BN, int OUT>
__device__ __forceinline__ void epilogue_tma(const CUtensorMap *tmC, uint32_t t_row, uint8_t *bufs,
                                             int &buf, int lane, int row0, int n0, int M,
                                             int N) {
  constexpr int OUT_COLS = OUT == GEMM_F32 ? 32 : 64;  // columns per 128-byte staging row
  const bool rows_in = row0 < M;
#pragma unroll 1
  for (int c0 = 0; c0 < BN; c0 += OUT_COLS) {
    uint32_t r0[32], r1[32];
    tmem_ld_32x32b_x32(t_row + c0, r0);
    if (OUT_COLS == 64) tmem_ld_32x32b_x32(t_row + c0 + 32, r1);
    tmem_wait_ld();
    if (!rows_in || n0 + c0 >= N) continue;  // warp-uniform: nothing of this box is in C
    uint8_t *sb = bufs + buf * kStoreBufBytes;
    if (lane == 0) bulk_wait_group_read<1>();  // the store that last used `sb` has read it
    __syncwarp();
    const uint32_t row_addr = smem_u32(sb) + lane * kRowBytes;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      uint32_t w0, w1, w2, w3;
      if (OUT == GEMM_F32) {
        w0 = r0[ch * 4 + 0], w1 = r0[ch * 4 + 1], w2 = r0[ch * 4 + 2], w3 = r0[ch * 4 + 3];
      } else {
        const int c = (ch & 3) * 8;
        const uint32_t *r = ch < 4 ? r0 : r1;
        w0 = pack2<OUT>(r[c + 0], r[c + 1]);
        w1 = pack2<OUT>(r[c + 2], r[c + 3]);
        w2 = pack2<OUT>(r[c + 4], r[c + 5]);
        w3 = pack2<OUT>(r[c + 6], r[c + 7]);
      }
      const uint32_t dst = row_addr + ((ch ^ (lane & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(w0), "r"(w1),
                   "r"(w2), "r"(w3)
                   : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmC, smem_u32(sb), n0 + c0, row0);
      bulk_commit_group();
    }
    buf ^= 1;
  }
}

// Epilogue, direct form for a C that TMA cannot address (misaligned base or ldc): each
// lane owns one row and writes its in-range columns with plain stores.
template <int BN, int OUT>
__device__ __forceinline__ void epilogue_direct(const TcParams &p, uint32_t t_row, int row, int n0) {
  using T = typename std::conditional<OUT == GEMM_F32, float,
            typename std::conditional<OUT == GEMM_BF16, __nv_bfloat16, __half>::type>::type;
#pragma unroll 1
  for (int c0 = 0; c0 < BN; c0 += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_row + c0, r);
    tmem_wait_ld();
    const int col = n0 + c0;
    if (row >= p.M || col >= p.N) continue;
    T *dst = reinterpret_cast<T *>(p.C) + static_cast<int64_t>(row) * p.ldc + col;
    const int n = min(32, p.N - col);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      if (j < n) {
        const float v = __uint_as_float(r[j]);
        if (OUT == GEMM_F32) {
          reinterpret_cast<float *>(dst)[j] = v;
        } else if (OUT == GEMM_BF16) {
          reinterpret_cast<__nv_bfloat16 *>(dst)[j] = __float2bfloat16_rn(v);
        } else {
          reinterpret_cast<__half *>(dst)[j] = __float2half_rn(v);
        }
      }
    }
  }
}

template <int ESIZE, bool A_MN, bool B_MN, int BN>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                   const __grid_constant__ CUtensorMap tmC, const TcParams p) {
  using G = Cfg<ESIZE, A_MN, B_MN, BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + G::BAR_OFFSET);
  uint64_t *empty = full + G::STAGES;
  uint64_t *tmem_full = empty + G::STAGES;
  uint64_t *tmem_empty = tmem_full + 2;
  uint64_t *drain = tmem_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], kEpiWarps * 32);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if (p.tma_store) prefetch_tensormap(&tmC);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), G::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};
  const int num_tiles = p.tiles_m * p.tiles_n;
  uint32_t issued = 0;  // stage fills issued by the producer lane

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = (p.debug_flags & kDebugStallProducer) == 0;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        int pm, pn;
        tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, pm, pn);
        const int m0 = pm * G::BM, n0 = pn * BN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, wd)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], G::STAGE_BYTES);
          const uint32_t a_dst = smem_u32(smem + stage * G::STAGE_BYTES);
          const uint32_t b_dst = a_dst + G::A_BYTES;
          const uint32_t fb = smem_u32(&full[stage]);
          const int k0 = kb * G::BK;
          if (A_MN) {
#pragma unroll
            for (int q = 0; q < G::BM / G::PANEL; ++q)
              tma_load_2d(a_dst + q * G::PANEL_BYTES, &tmA, fb, m0 + q * G::PANEL, k0);
          } else {
            tma_load_2d(a_dst, &tmA, fb, k0, m0);
          }
          if (B_MN) {
#pragma unroll
            for (int q = 0; q < BN / G::PANEL; ++q)
              tma_load_2d(b_dst + q * G::PANEL_BYTES, &tmB, fb, n0 + q * G::PANEL, k0);
          } else {
            tma_load_2d(b_dst, &tmB, fb, k0, n0);
          }
          ++issued;
          if (++stage == G::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        if (!mbar_wait(&tmem_empty[acc], acc_phase ^ 1, wd)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < p.k_blocks; ++kb) {
          if (!mbar_wait(&full[stage], phase, wd)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * G::STAGE_BYTES);
          const uint32_t b_base = a_base + G::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < G::K_STEPS; ++kk) {
            // K-major: step 32 bytes along the swizzled row; MN-major: step UMMA_K rows.
            const uint64_t ad =
                A_MN ? sdesc_sw128(a_base + kk * G::UMMA_K * kRowBytes, G::PANEL_BYTES, 1024)
                     : sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd =
                B_MN ? sdesc_sw128(b_base + kk * G::UMMA_K * kRowBytes, G::PANEL_BYTES, 1024)
                     : sdesc_sw128(b_base + kk * 32, 16, 1024);
            const uint32_t accumulate = (kb | kk) != 0;
            if (ESIZE == 2)
              mma_f16(d_tmem, ad, bd, p.idesc, accumulate);
            else
              mma_tf32(d_tmem, ad, bd, p.idesc, accumulate);
          }
          mma_commit(&empty[stage]);  // frees the stage once these MMAs have read it
          if (++stage == G::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit(&tmem_full[acc]);  // accumulator complete once every MMA above is done
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      // Every MMA issued above must finish before TMEM is released.
      mma_commit(drain);
      drain_wait(drain, 0, p.timeout_ns);
    }
    __syncwarp();
  } else {
    // --------------------------------------------------------------- epilogue
    const int quarter = warp & 3;  // TMEM lanes this warp may access: 32*quarter ...
    uint8_t *bufs = smem + G::EPI_OFFSET + (warp - 2) * 2 * kStoreBufBytes;
    int buf = 0;
    uint32_t acc = 0, acc_phase = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x) {
      bool ok = mbar_wait(&tmem_full[acc], acc_phase, wd);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      int pm, pn;
      tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, pm, pn);
      const int row0 = pm * G::BM + quarter * 32;
      const int n0 = pn * BN;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN;
      if (p.tma_store) {
        if (p.out_dtype == GEMM_BF16)
          epilogue_tma<BN, GEMM_BF16>(&tmC, t_row, bufs, buf, lane, row0, n0, p.M, p.N);
        else if (p.out_dtype == GEMM_F16)
          epilogue_tma<BN, GEMM_F16>(&tmC, t_row, bufs, buf, lane, row0, n0, p.M, p.N);
        else
          epilogue_tma<BN, GEMM_F32>(&tmC, t_row, bufs, buf, lane, row0, n0, p.M, p.N);
      } else {
        if (p.out_dtype == GEMM_BF16)
          epilogue_direct<BN, GEMM_BF16>(p, t_row, row0 + lane, n0);
        else if (p.out_dtype == GEMM_F16)
          epilogue_direct<BN, GEMM_F16>(p, t_row, row0 + lane, n0);
        else
          epilogue_direct<BN, GEMM_F32>(p, t_row, row0 + lane, n0);
      }
      tc_fence_before();
      mbar_arrive(&tmem_empty[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (lane == 0) bulk_wait_group<0>();  // C writes complete before the CTA exits
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, G::TMEM_COLS);
  }
  if (warp == 0 && lane == 0 && *abort_flag) {
    // After an abort, let every copy already issued land before the CTA exits: the last
    // fill of stage s is fill number f (f % STAGES == s), completing parity (f/STAGES)&1.
    for (uint32_t s = 0; s < G::STAGES && s < issued; ++s) {
      const uint32_t f = s + G::STAGES * ((issued - 1 - s) / G::STAGES);
      drain_wait(&full[s], (f / G::STAGES) & 1, p.timeout_ns);
    }
  }
}

template <int ESIZE, bool A_MN, bool B_MN, int BN>
cudaError_t launch_one(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                       const TcParams &p, int grid, cudaStream_t s) {
  using G = Cfg<ESIZE, A_MN, B_MN, BN>;
  auto kernel = tc_gemm_kernel<ESIZE, A_MN, B_MN, BN>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  kernel<<<grid, kThreads, G::SMEM_BYTES, s>>>(tmA, tmB, tmC, p);
  return cudaGetLastError();
}

template <int ESIZE, int BN>
cudaError_t launch_majors(const TcVariant &v, const CUtensorMap &tmA, const CUtensorMap &tmB,
                          const CUtensorMap &tmC, const TcParams &p, int grid, cudaStream_t s) {
  if (!v.a_mn && !v.b_mn) return launch_one<ESIZE, false, false, BN>(tmA, tmB, tmC, p, grid, s);
  if (!v.a_mn && v.b_mn) return launch_one<ESIZE, false, true, BN>(tmA, tmB, tmC, p, grid, s);
  if (v.a_mn && !v.b_mn) return launch_one<ESIZE, true, false, BN>(tmA, tmB, tmC, p, grid, s);
  return launch_one<ESIZE, true, true, BN>(tmA, tmB, tmC, p, grid, s);
}

}  // namespace

int tc_stages(const TcVariant &v) { return v.block_n >= 256 ? 4 : 6; }

size_t tc_smem_bytes(const TcVariant &v) {
  if (v.block_n == 256) return Cfg<2, false, false, 256>::SMEM_BYTES;
  return Cfg<2, false, false, 128>::SMEM_BYTES;
}

cudaError_t tc_launch(const TcVariant &v, const CUtensorMap &tmA, const CUtensorMap &tmB,
                      const CUtensorMap &tmC, const TcParams &p, int grid, cudaStream_t s) {
  if (v.esize == 2 && v.block_n == 256) return launch_majors<2, 256>(v, tmA, tmB, tmC, p, grid, s);
  if (v.esize == 4 && v.block_n == 256) return launch_majors<4, 256>(v, tmA, tmB, tmC, p, grid, s);
  if (v.esize == 2 && v.block_n == 128) return launch_majors<2, 128>(v, tmA, tmB, tmC, p, grid, s);
  if (v.esize == 4 && v.block_n == 128) return launch_majors<4, 128>(v, tmA, tmB, tmC, p, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace gemm_gb300
