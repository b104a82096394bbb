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
#include "tc_common.cuh"

namespace gemm_gb300 {
namespace {

using namespace tc;

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
  // The prologue above may overlap the previous kernel on the stream; global memory only
  // from here on.
  grid_dependency_wait();
  grid_launch_dependents();
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};
  const int num_tiles = p.tiles_m * p.tiles_n;
  uint32_t issued = 0;  // stage fills issued by the producer lane

  if (warp == 0) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      bool ok = (p.debug_flags & kDebugStallProducer) == 0;
      // test hook: the loader stops after this many stage fills (-1: never)
      const int stop_after = stall_after_fills(p.debug_flags & ~kDebugStallRank1, 0);
      // Operand tiles stay in L2 longest, unless only one tile row or column reads them.
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t pol_a = (p.l2_once & kL2OnceA) ? l2_policy_evict_first() : keep;
      const uint64_t pol_b = (p.l2_once & kL2OnceB) ? l2_policy_evict_first() : keep;
      for (int tile = blockIdx.x; ok && tile < num_tiles; tile += gridDim.x) {
        int pm, pn;
        tile_coords(tile, p.tiles_m, p.tiles_n, p.group_m, pm, pn);
        const int m0 = pm * G::BM, n0 = pn * BN;
        // the tile's K-loop may start at any K-block: the same K-blocks are summed
        const int rot =
            p.k_rotate ? static_cast<int>(static_cast<int64_t>(tile) * p.k_rotate % p.k_blocks) : 0;
        for (int kb_i = 0; kb_i < p.k_blocks; ++kb_i) {
          const int kb = kb_i + rot < p.k_blocks ? kb_i + rot : kb_i + rot - p.k_blocks;
          if (stop_after >= 0 && issued >= static_cast<uint32_t>(stop_after)) {
            ok = false;  // test hook: the loader stops here, copies still in flight
            break;
          }
          if (!mbar_wait(&empty[stage], phase ^ 1, wd)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], G::STAGE_BYTES);
          const uint32_t a_dst = smem_u32(smem + stage * G::STAGE_BYTES);
          const uint32_t b_dst = a_dst + G::A_BYTES;
          const uint32_t fb = smem_u32(&full[stage]);
          const int k0 = kb * G::BK;
          if (A_MN && (p.mn_3d & kMn3dA)) {
            tma_load_3d_hint(a_dst, &tmA, fb, 0, k0, m0 / G::PANEL, pol_a);
          } else if (A_MN) {
#pragma unroll
            for (int q = 0; q < G::BM / G::PANEL; ++q)
              tma_load_2d_hint(a_dst + q * G::PANEL_BYTES, &tmA, fb, m0 + q * G::PANEL, k0, pol_a);
          } else {
            tma_load_2d_hint(a_dst, &tmA, fb, k0, m0, pol_a);
          }
          if (B_MN && (p.mn_3d & kMn3dB)) {
            tma_load_3d_hint(b_dst, &tmB, fb, 0, k0, n0 / G::PANEL, pol_b);
          } else if (B_MN) {
#pragma unroll
            for (int q = 0; q < BN / G::PANEL; ++q)
              tma_load_2d_hint(b_dst + q * G::PANEL_BYTES, &tmB, fb, n0 + q * G::PANEL, k0, pol_b);
          } else {
            tma_load_2d_hint(b_dst, &tmB, fb, k0, n0, pol_b);
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
                A_MN ? sdesc_sw128(a_base + kk * G::UMMA_K * kRowBytes, G::PANEL_BYTES,
                                  sdesc_mn_sbo<ESIZE>(), sdesc_mode<ESIZE, true>())
                     : sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd =
                B_MN ? sdesc_sw128(b_base + kk * G::UMMA_K * kRowBytes, G::PANEL_BYTES,
                                  sdesc_mn_sbo<ESIZE>(), sdesc_mode<ESIZE, true>())
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
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see grid_dependency_wait
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = G::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmC, p);
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

int tc_stages(const TcVariant &v) {
  if (v.pair) return (v.block_n >= 256 ? 6 : 8) / v.kps;
  return v.block_n >= 256 ? 4 : 6;
}

cudaError_t tc_launch(const TcVariant &v, const CUtensorMap &tmA, const CUtensorMap &tmB,
                      const CUtensorMap &tmC, const CUtensorMap &tmP, const TcParams &p, int grid,
                      cudaStream_t s) {
  if (v.exact || v.f16acc) return tc_chunk_launch(v.f16acc, tmA, tmB, tmC, tmP, p, grid, s);
  if (v.pair) return tc2_launch(v, tmA, tmB, tmC, tmP, p, grid, s);
  if (v.esize == 2 && v.block_n == 256) return launch_majors<2, 256>(v, tmA, tmB, tmC, p, grid, s);
  if (v.esize == 4 && v.block_n == 256) return launch_majors<4, 256>(v, tmA, tmB, tmC, p, grid, s);
  if (v.esize == 2 && v.block_n == 128) return launch_majors<2, 128>(v, tmA, tmB, tmC, p, grid, s);
  if (v.esize == 4 && v.block_n == 128) return launch_majors<4, 128>(v, tmA, tmB, tmC, p, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace gemm_gb300
