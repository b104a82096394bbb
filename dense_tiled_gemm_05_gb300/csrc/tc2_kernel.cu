// tc2_kernel.cu -- the tensor-core blocked GEMM on CTA pairs (cta_group::2, two SMs).
//
// Same computation and roles as tc_kernel.cu ("Chapter 13: The Blocked Matmul Kernel",
// section 13.1: a grid of output tiles, each walking its K-chunks into an fp32 accumulator
// initialised once; section 13.2's masks from the TMA unit's zero fill and clipped stores),
// but each output tile is 256 x 256 and is computed by a cluster of two CTAs on two SMs:
//   * each CTA TMA-loads its own 128 rows of A and its own 128 columns of B per K-chunk
//     into its shared memory and signals the leader CTA's full barrier;
//   * the leader's MMA thread issues tcgen05.mma.cta_group::2 (M = 256, N = 256): the
//     hardware reads A and B halves from both CTAs' shared memory and writes rows 0-127 of
//     the accumulator to the leader's TMEM and rows 128-255 to the peer's TMEM;
//   * commits multicast to the barriers of both CTAs (stage free; accumulator ready);
//   * both CTAs' epilogue warps drain their own TMEM and release the leader's TMEM-empty
//     barrier (the peer arrives remotely).
// Each SM therefore streams half as much B per flop as the single-CTA 128 x 256 tile, and
// each output tile needs half the L2 traffic per flop.
//
// A stage holds KPS consecutive 128-byte K-blocks of each K-major operand (KPS = 1 or 2):
// with 2, every row of A and B is fetched 256 contiguous bytes at a time, which keeps more
// of each DRAM page's bytes in one request stream when the product is bandwidth-bound.
//
// Schedule options carried in TcParams: a CTA may load fewer than 128 rows of A
// (cta_rows; the surplus accumulator lanes are never stored); an operand read by one tile
// row or column only is loaded as first to evict from L2, and every piece of a K-loop
// then starts at a staggered K-block (k_rotate); pieces of tiles split along K hand their
// fp32 sums to the tile's owner through the workspace (sk_schedule.h).
#include "tc_common.cuh"

namespace gemm_gb300 {
namespace {

using namespace tc;

template <int ESIZE, bool A_MN, bool B_MN, int BN_, int KPS = 1>
struct Cfg2 {
  static constexpr int BM = kTcBlockM;             // rows per CTA (256 per pair)
  static constexpr int BN = BN_;                   // columns per pair tile (256 or 128)
  static constexpr int BN_HALF = BN / 2;           // B columns loaded by each CTA
  static constexpr int BOX_K = kRowBytes / ESIZE;  // K elements per 128-byte K-block
  static constexpr int BK = KPS * BOX_K;           // K elements per stage
  static constexpr int UMMA_K = 32 / ESIZE;        // K elements per tcgen05.mma
  static constexpr int K_STEPS = BK / UMMA_K;
  static constexpr int BOX_STEPS = BOX_K / UMMA_K;  // MMAs per K-block
  static constexpr int PANEL = kRowBytes / ESIZE;  // M/N elements per 128-byte row (MN-major)
  static constexpr int PANEL_BYTES = BK * kRowBytes;
  static constexpr int A_BYTES = BM * BK * ESIZE;
  static constexpr int B_BYTES = BN_HALF * BK * ESIZE;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // per CTA
  static constexpr int A_BOX_BYTES = BM * kRowBytes;       // one K-block of A
  static constexpr int B_BOX_BYTES = BN_HALF * kRowBytes;  // one K-block of B
  static constexpr int STAGES = (BN >= 256 ? 6 : 8) / KPS;
  static constexpr int EPI_OFFSET = STAGES * STAGE_BYTES;
  static constexpr int EPI_BYTES = kEpiWarps * 2 * kStoreBufBytes;
  static constexpr int BAR_OFFSET = EPI_OFFSET + EPI_BYTES;
  static constexpr int OWNER_SLICE = 48 * 1024;     // stage bytes an owner warp borrows
  static constexpr int PART_BYTES = BN * 32 * 4;    // one partial's 32 rows, fp32
  static constexpr int PART_BUFS = OWNER_SLICE / PART_BYTES;  // partial loads in flight
  // + one partial-load barrier per buffer of each epilogue warp
  static constexpr int NUM_BARS = 2 * STAGES + 5 + kEpiWarps * PART_BUFS;
  // + TMEM address, abort flag and the four teardown words (see `xs` in the kernel)
  static constexpr int SMEM_BYTES = BAR_OFFSET + NUM_BARS * 8 + 32 + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(kEpiWarps * OWNER_SLICE <= STAGES * STAGE_BYTES, "owner slices fit the stages");
  static_assert(PART_BUFS >= 1 && PART_BUFS <= 3, "a warp's partial rows fit its slice");
  static_assert(KPS == 1 || (!A_MN && !B_MN), "wide stages for K-major operands only");
};

// Wait on a barrier of the operand ring (stage full, stage empty). Their arrivals come
// from the async units (TMA copies completing, tcgen05.commit), and what the waiting thread
// does next is issue more async work (MMAs reading the stage, copies refilling it), so an
// acquire at CTA scope is enough; at cluster scope each wait costs more. Measured on one
// GB300 (interleaved, order rotated, CUDA events): bf16 4096^3 93.0 -> 90.9 us,
// 2048^2 x 8192 48.2 -> 46.5, 8192^3 -1 %; tf32 unchanged.
__device__ __forceinline__ bool ring_wait(uint64_t *bar, uint32_t parity, const Watchdog &wd) {
  return mbar_wait(bar, parity, wd);
}

template <int ESIZE, bool A_MN, bool B_MN, int BN, int KPS>
__global__ void __launch_bounds__(kThreads, 1)
    tc2_gemm_kernel(const __grid_constant__ CUtensorMap tmA,
                    const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC,
                    const __grid_constant__ CUtensorMap tmP, const TcParams p) {
  using G = Cfg2<ESIZE, A_MN, B_MN, BN, KPS>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + G::BAR_OFFSET);
  uint64_t *empty = full + G::STAGES;
  uint64_t *tmem_full = empty + G::STAGES;
  uint64_t *tmem_empty = tmem_full + 2;
  uint64_t *drain = tmem_empty + 2;
  uint64_t *part_bar = drain + 1;  // [kEpiWarps][PART_BUFS]: owner warps' partial loads
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(part_bar + kEpiWarps * G::PART_BUFS);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
  // Teardown words: [0] stage fills this CTA's loader issued, [1] fills the MMA issuer
  // consumed (leader), [2] fills the peer's loader issued (the peer writes it into the
  // leader), [3] whether the other CTA of the pair aborted (written by that CTA).
  volatile uint32_t *xs = reinterpret_cast<volatile uint32_t *>(tmem_slot + 2);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();  // 0: leader (issues the MMAs), 1: peer
  const bool leader = rank == 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(&full[s], 1);   // the leader's arrive.expect_tx (bytes of both CTAs)
      mbar_init(&empty[s], 1);  // the leader's multicast commit
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);               // the leader's multicast commit
      mbar_init(&tmem_empty[b], 2 * kEpiWarps);  // one arrive per epilogue warp, both CTAs
    }
    mbar_init(drain, 1);
    for (int w = 0; w < kEpiWarps * G::PART_BUFS; ++w) mbar_init(&part_bar[w], 1);
    *abort_flag = 0;
    for (int i = 0; i < 4; ++i) xs[i] = 0;
    fence_barrier_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if (p.tma_store) prefetch_tensormap(&tmC);
  }
  if (warp == 1) {
    tmem_alloc_pair(smem_u32(tmem_slot), G::TMEM_COLS);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  cluster_sync();  // barriers of both CTAs initialised; TMEM allocated in both
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Everything above touches only this CTA's own resources, so it may overlap the end of
  // the previous kernel on the stream; from here on global memory is read and written.
  grid_dependency_wait();
  grid_launch_dependents();
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};
  const int cluster_id = blockIdx.x / 2;
  const int num_clusters = gridDim.x / 2;
  // Whole tiles round-robin over the clusters, then the split-K share of the last rounds.
  const SkSchedule sched = sk_make(p.tiles_m * p.tiles_n, p.k_blocks, num_clusters, p.sk_dp_tiles);
  const bool split = p.sk_dp_tiles < p.tiles_m * p.tiles_n;
  const int epoch = split ? sk_epoch_begin(p.sk_epoch_word) : 0;

  if (warp == 0) {
    // ------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = (p.debug_flags & kDebugStallProducer) == 0;
      const int stop_after = stall_after_fills(p.debug_flags, static_cast<int>(rank));
      // Operand tiles stay in L2 longest, unless only one tile row or column reads them.
      const uint64_t keep = l2_policy_evict_last();
      const uint64_t pol_a = (p.l2_once & kL2OnceA) ? l2_policy_evict_first() : keep;
      const uint64_t pol_b = (p.l2_once & kL2OnceB) ? l2_policy_evict_first() : keep;
      // This CTA's rows of the tile (fewer than the MMA's 128 under GEMM_OPT_TILE_ROWS)
      // and the bytes both CTAs load per stage.
      const int rows = p.cta_rows;
      const uint32_t stage_tx = 2u * static_cast<uint32_t>(rows * G::BK * ESIZE + G::B_BYTES);
      WorkIter work(sched, cluster_id);
      SkSegment seg;
      while (ok && work.next(seg)) {
        int pm, pn;
        tile_coords(seg.tile, p.tiles_m, p.tiles_n, p.group_m, pm, pn);
        const int m0 = pm * (2 * rows) + static_cast<int>(rank) * rows;
        const int n0 = pn * G::BN + static_cast<int>(rank) * G::BN_HALF;
        // A piece may walk its K-blocks from any one of them, wrapping around: its sum
        // takes the same set of K-blocks.
        const int len = seg.kb_end - seg.kb_begin;
        const int rot =
            p.k_rotate ? static_cast<int>(static_cast<int64_t>(seg.tile) * p.k_rotate % len) : 0;
        for (int i = 0; i < len; ++i) {
          const int kb = seg.kb_begin + (i + rot < len ? i + rot : i + rot - len);
          if (stop_after >= 0 && issued >= static_cast<uint32_t>(stop_after)) {
            ok = false;  // test hook: this loader stops here, copies still in flight
            break;
          }
          if (!ring_wait(&empty[stage], phase ^ 1, wd)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], stage_tx);
          const uint32_t a_dst = smem_u32(smem + stage * G::STAGE_BYTES);
          const uint32_t b_dst = a_dst + G::A_BYTES;
          const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);  // the leader's barrier
          const int k0 = kb * G::BK;
          if (A_MN && (p.mn_3d & kMn3dA)) {
            tma_load_3d_pair_hint(a_dst, &tmA, fb, 0, k0, m0 / G::PANEL, pol_a);
          } else if (A_MN) {
#pragma unroll
            for (int q = 0; q < G::BM / G::PANEL; ++q)
              tma_load_2d_pair_hint(a_dst + q * G::PANEL_BYTES, &tmA, fb, m0 + q * G::PANEL, k0,
                                    pol_a);
          } else {
#pragma unroll
            for (int j = 0; j < KPS; ++j)
              tma_load_2d_pair_hint(a_dst + j * G::A_BOX_BYTES, &tmA, fb, k0 + j * G::BOX_K, m0,
                                    pol_a);
          }
          if (B_MN && (p.mn_3d & kMn3dB)) {
            tma_load_3d_pair_hint(b_dst, &tmB, fb, 0, k0, n0 / G::PANEL, pol_b);
          } else if (B_MN) {
#pragma unroll
            for (int q = 0; q < G::BN_HALF / G::PANEL; ++q)
              tma_load_2d_pair_hint(b_dst + q * G::PANEL_BYTES, &tmB, fb, n0 + q * G::PANEL, k0,
                                    pol_b);
          } else {
#pragma unroll
            for (int j = 0; j < KPS; ++j)
              tma_load_2d_pair_hint(b_dst + j * G::B_BOX_BYTES, &tmB, fb, k0 + j * G::BOX_K, n0,
                                    pol_b);
          }
          ++issued;
          if (++stage == G::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      xs[0] = issued;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------ MMA issuer (leader)
    if (leader && lane == 0) {
      uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, consumed = 0;
      bool ok = true;
      WorkIter work(sched, cluster_id);
      SkSegment seg;
      while (ok && work.next(seg)) {
        if (!mbar_wait_cluster(&tmem_empty[acc], acc_phase ^ 1, wd)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * G::BN;
        for (int kb = seg.kb_begin; kb < seg.kb_end; ++kb) {
          if (!ring_wait(&full[stage], phase, wd)) {
            ok = false;
            break;
          }
          ++consumed;
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * G::STAGE_BYTES);
          const uint32_t b_base = a_base + G::A_BYTES;
#pragma unroll
          for (int kk = 0; kk < G::K_STEPS; ++kk) {
            // K-major: K-block kk / BOX_STEPS of the stage, 32 bytes per MMA inside it
            const uint32_t a_k = (kk / G::BOX_STEPS) * G::A_BOX_BYTES + (kk % G::BOX_STEPS) * 32;
            const uint32_t b_k = (kk / G::BOX_STEPS) * G::B_BOX_BYTES + (kk % G::BOX_STEPS) * 32;
            const uint64_t ad =
                A_MN ? sdesc_sw128(a_base + kk * G::UMMA_K * kRowBytes, G::PANEL_BYTES,
                                  sdesc_mn_sbo<ESIZE>(), sdesc_mode<ESIZE, true>())
                     : sdesc_sw128(a_base + a_k, 16, 1024);
            const uint64_t bd =
                B_MN ? sdesc_sw128(b_base + kk * G::UMMA_K * kRowBytes, G::PANEL_BYTES,
                                  sdesc_mn_sbo<ESIZE>(), sdesc_mode<ESIZE, true>())
                     : sdesc_sw128(b_base + b_k, 16, 1024);
            const uint32_t accumulate = (kb != seg.kb_begin) || kk != 0;
            if (ESIZE == 2)
              mma_f16_pair(d_tmem, ad, bd, p.idesc, accumulate);
            else
              mma_tf32_pair(d_tmem, ad, bd, p.idesc, accumulate);
          }
          mma_commit_pair_multicast(&empty[stage], 0x3);  // stage free in both CTAs
          if (++stage == G::STAGES) {
            stage = 0;
            phase ^= 1;
          }
        }
        if (!ok) break;
        mma_commit_pair_multicast(&tmem_full[acc], 0x3);  // accumulator ready in both CTAs
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      mma_commit_pair(drain);  // every MMA issued above completes before TMEM is released
      drain_wait(drain, 0, p.timeout_ns);
      xs[1] = consumed;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue (both CTAs)
    const int quarter = warp & 3;
    uint8_t *bufs = smem + G::EPI_OFFSET + (warp - 2) * 2 * kStoreBufBytes;
    int buf = 0;
    uint32_t acc = 0, acc_phase = 0;
    WorkIter work(sched, cluster_id);
    SkSegment seg;
    const int e = warp - 2;       // epilogue warp index
    uint32_t part_phase = 0;      // parities of this warp's partial-load barriers (bit b)
    bool ok = true;
    while (ok && work.next(seg)) {
      ok = mbar_wait_cluster(&tmem_full[acc], acc_phase, wd);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      int pm, pn;
      tile_coords(seg.tile, p.tiles_m, p.tiles_n, p.group_m, pm, pn);
      const int row0 = pm * (2 * p.cta_rows) + static_cast<int>(rank) * p.cta_rows + quarter * 32;
      // Accumulator lanes of this warp that hold rows of the tile (all 32 unless the tile
      // is shorter than the MMA).
      const int valid = p.cta_rows - quarter * 32;
      const int n0 = pn * G::BN;
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + acc * G::BN;
      // First row of this warp's 32 rows in worker w's partial tile (row-major, BN columns).
      auto part_row0 = [&](int w) { return (w * 2 + static_cast<int>(rank)) * G::BM + quarter * 32; };
      if (seg.role == kSegPartial) {
        // Split-K piece without its tile's last K-block: its fp32 sum goes to this worker's
        // workspace entry by TMA store; the flag tells the tile's owner it is in memory.
        epilogue_tma<G::BN, GEMM_F32>(&tmP, t_row, bufs, buf, lane, part_row0(cluster_id), 0,
                                      INT32_MAX, G::BN);
        if (lane == 0) {
          bulk_wait_group<0>();  // the partial's writes are complete
          fence_proxy_async_global();
          st_release_gpu(p.sk_flags + (cluster_id * 2 + rank) * 4 + quarter, epoch);
        }
        __syncwarp();
      } else {
        if (seg.role == kSegOwner) {
          // The start of this tile was computed by workers first_src..last_src (all numbered
          // below this one): add their partials into the accumulator in increasing worker
          // order (a fixed order). The owner piece is its worker's last, so the pipeline
          // stages are idle and each epilogue warp borrows a slice of them: up to PART_BUFS
          // partials are loaded ahead of the one being added.
          uint8_t *slice = smem + e * G::OWNER_SLICE;
          uint64_t *bars = part_bar + e * G::PART_BUFS;
          const int nsrc = seg.last_src - seg.first_src + 1;
          // Wait for partial i's flag, then load it into buffer i % PART_BUFS.
          int fetched = 0, added = 0;  // partial loads issued, and waited for
          auto fetch = [&](int i) {
            const int w = seg.first_src + i;
            bool f = wait_flag(p.sk_flags + (w * 2 + rank) * 4 + quarter, epoch, wd);
            f = __all_sync(0xffffffffu, f);
            if (!f) return false;
            fence_proxy_async_global();
            if (lane == 0) {
              const int b = i % G::PART_BUFS;
              uint8_t *buf = slice + b * G::PART_BYTES;
              mbar_arrive_expect_tx(&bars[b], G::PART_BYTES);
#pragma unroll
              for (int c = 0; c < G::BN / 32; ++c)
                tma_load_2d(smem_u32(buf + c * kStoreBufBytes), &tmP, smem_u32(&bars[b]), c * 32,
                            part_row0(w));
            }
            ++fetched;
            return true;
          };
          for (int i = 0; ok && i < nsrc && i < G::PART_BUFS; ++i) ok = fetch(i);
          for (int i = 0; ok && i < nsrc; ++i) {
            const int b = i % G::PART_BUFS;
            ok = mbar_wait(&bars[b], (part_phase >> b) & 1u, wd);
            ok = __all_sync(0xffffffffu, ok);
            if (!ok) break;
            part_phase ^= 1u << b;
            ++added;
            add_partial_into_tmem<G::BN>(t_row, slice + b * G::PART_BYTES, lane);
            if (i + G::PART_BUFS < nsrc) {
              __syncwarp();               // every lane has read buffer b
              fence_proxy_async_smem();   // before the TMA unit writes it again
              ok = fetch(i + G::PART_BUFS);
            }
          }
          if (!ok) {
            // Partial loads already issued may still be landing in this warp's slice: let
            // them complete (each buffer holds at most one) before the CTA can leave.
            if (lane == 0)
              for (int i = added; i < fetched; ++i) {
                const int b = i % G::PART_BUFS;
                drain_wait(&bars[b], (part_phase >> b) & 1u, p.timeout_ns);
                part_phase ^= 1u << b;
              }
            __syncwarp();
            break;
          }
        }
        if (valid <= 0) {
          // no row of the tile in this warp's lanes
        } else if (p.tma_store && valid >= 32) {
          if (p.out_dtype == GEMM_BF16)
            epilogue_tma<G::BN, GEMM_BF16>(&tmC, t_row, bufs, buf, lane, row0, n0, p.M, p.N);
          else if (p.out_dtype == GEMM_F16)
            epilogue_tma<G::BN, GEMM_F16>(&tmC, t_row, bufs, buf, lane, row0, n0, p.M, p.N);
          else
            epilogue_tma<G::BN, GEMM_F32>(&tmC, t_row, bufs, buf, lane, row0, n0, p.M, p.N);
        } else {
          // plain stores; lanes past the tile's last row store nothing (row beyond C)
          const int row = lane < valid ? row0 + lane : INT32_MAX;
          if (p.out_dtype == GEMM_BF16)
            epilogue_direct<G::BN, GEMM_BF16>(p, t_row, row, n0);
          else if (p.out_dtype == GEMM_F16)
            epilogue_direct<G::BN, GEMM_F16>(p, t_row, row, n0);
          else
            epilogue_direct<G::BN, GEMM_F32>(p, t_row, row, n0);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[acc]), 0));
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1;
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  __syncthreads();
  // Tell the other CTA whether this one aborted, and the leader how many stage fills the
  // peer's loader issued (the peer's copies complete on the leader's barriers).
  if (threadIdx.x == 0) {
    st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t *>(&xs[3])), rank ^ 1u),
                          *abort_flag ? 1u : 0u);
    if (!leader) st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t *>(&xs[2])), 0), xs[0]);
  }
  tc_fence_before();
  cluster_sync();  // both CTAs done, all MMAs drained; abort states exchanged
  if (*abort_flag || xs[3]) {
    // After an abort, neither CTA leaves while a copy it issued may still land in its
    // shared memory: the leader accounts for every outstanding fill and waits for it.
    if (leader && threadIdx.x == 0)
      drain_pair_fills<G::STAGES>(full, xs[1], xs[0], xs[2],
                                  static_cast<uint32_t>(p.cta_rows * G::BK * ESIZE + G::B_BYTES),
                                  p.timeout_ns);
    cluster_sync();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, G::TMEM_COLS);
  }
  if (split && threadIdx.x == 0) sk_epoch_end(p.sk_epoch_word, epoch);
}

template <int ESIZE, bool A_MN, bool B_MN, int BN, int KPS = 1>
cudaError_t launch_pair(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                        const CUtensorMap &tmP, const TcParams &p, int grid, cudaStream_t s) {
  using G = Cfg2<ESIZE, A_MN, B_MN, BN, KPS>;
  auto kernel = tc2_gemm_kernel<ESIZE, A_MN, B_MN, BN, KPS>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // The prologue (barriers, TMEM, tensor-map prefetch) may overlap the previous kernel's
  // tail; the kernel waits for it before touching global memory.
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = G::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, tmA, tmB, tmC, tmP, p);
}

template <int ESIZE, int BN>
cudaError_t launch_pair_majors(const TcVariant &v, const CUtensorMap &tmA, const CUtensorMap &tmB,
                               const CUtensorMap &tmC, const CUtensorMap &tmP, const TcParams &p,
                               int grid, cudaStream_t s) {
  if (!v.a_mn && !v.b_mn) return launch_pair<ESIZE, false, false, BN>(tmA, tmB, tmC, tmP, p, grid, s);
  if (!v.a_mn && v.b_mn) return launch_pair<ESIZE, false, true, BN>(tmA, tmB, tmC, tmP, p, grid, s);
  if (v.a_mn && !v.b_mn) return launch_pair<ESIZE, true, false, BN>(tmA, tmB, tmC, tmP, p, grid, s);
  return launch_pair<ESIZE, true, true, BN>(tmA, tmB, tmC, tmP, p, grid, s);
}

}  // namespace

int tc2_max_active_clusters() {
  static int cached[64];  // per device; 0 = not queried yet
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  if (cached[dev] > 0) return cached[dev];
  using G = Cfg2<2, false, false, 256, 1>;
  auto kernel = tc2_gemm_kernel<2, false, false, 256, 1>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM_BYTES) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = G::SMEM_BYTES;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cached[dev] = n;
  return n;
}

cudaError_t tc2_launch(const TcVariant &v, const CUtensorMap &tmA, const CUtensorMap &tmB,
                       const CUtensorMap &tmC, const CUtensorMap &tmP, const TcParams &p, int grid,
                       cudaStream_t s) {
  if (v.kps == 2 && v.esize == 2 && !v.a_mn && !v.b_mn) {
    if (v.block_n == 256) return launch_pair<2, false, false, 256, 2>(tmA, tmB, tmC, tmP, p, grid, s);
    if (v.block_n == 128) return launch_pair<2, false, false, 128, 2>(tmA, tmB, tmC, tmP, p, grid, s);
    return cudaErrorInvalidValue;
  }
  if (v.esize == 2 && v.block_n == 256)
    return launch_pair_majors<2, 256>(v, tmA, tmB, tmC, tmP, p, grid, s);
  if (v.esize == 2 && v.block_n == 128)
    return launch_pair_majors<2, 128>(v, tmA, tmB, tmC, tmP, p, grid, s);
  if (v.esize == 4 && v.block_n == 256)
    return launch_pair_majors<4, 256>(v, tmA, tmB, tmC, tmP, p, grid, s);
  if (v.esize == 4 && v.block_n == 128)
    return launch_pair_majors<4, 128>(v, tmA, tmB, tmC, tmP, p, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace gemm_gb300
