// tc_chunk_kernel.cu -- tensor-core GEMMs whose accumulator lives in registers and takes
// the tensor cores' fp32 partial products one short K-chunk at a time (CTA pairs).
//
// Two modes share the kernel; both keep the tile structure of the blocked matmul of
// "Chapter 13: The Blocked Matmul Kernel", section 13.1 (the accumulator starts at zero once
// per tile, every K-chunk's partial product is added to it, the result is stored once),
// and both let the MMA issuer alternate between two TMEM accumulators, starting a fresh one
// every `chunk_steps` MMA instructions, while the epilogue warps add each finished chunk
// into their registers.
//
// * Exact fp32 ("Triton matmul", "Precision": fp32 inputs need an explicit choice between
//   tf32 and full fp32 accuracy) on the tf32 tensor cores: split_kernel.cu writes each
//   operand as [hi | lo], and the producer walks the K-blocks of
//   A' = [hi(A) | hi(A) | lo(A)] and B' = [hi(B) ; lo(B) ; hi(B)] by picking the part for
//   each, so that A' B' holds the three significant partial products of the split operands. The tensor cores' fp32
//   accumulation over a long K drifts (measured on GB300: 4e-6 of sum |a b| at K = 4096,
//   growing with K), so no TMEM accumulator runs over more than a short chunk, and the
//   chunks are summed in fp32 registers with ordinary IEEE adds; rounded once at the store.
//
// * fp16 accumulator (section 13.3, Worked Example 13.3.1): fp16 inputs, and an
//   accumulator held in fp16 that rounds after every K-chunk: each chunk's dot product
//   (fp32, from the tensor cores) is rounded to fp16 and added to the fp16 running total
//   with an fp16 add (round to nearest even). One chunk is a multiple of the 16-long K of
//   one tcgen05.mma.kind::f16.
//
// In exact mode the last, partly filled rounds of tiles may be split along K over all
// clusters (the schedule of sk_schedule.h, as in the CTA-pair kernel): a piece without its
// tile's last K-block stores its fp32 register sums to the handle's workspace and raises a
// flag; the piece holding the last K-block adds the lower-numbered workers' partials into
// its register sums in increasing worker order before storing. The fp16 accumulator never
// splits: its running total must see the chunks one after another.
//
// Roles (320 threads per CTA, clusters of two CTAs, 256 x 256 tile per cluster):
//   warp 0      TMA producer (both CTAs): 128 rows of A, 128 columns of B per 128-byte K-block;
//   warp 1      MMA issuer (leader CTA): tcgen05.mma.cta_group::2, M=256, N=256;
//   warps 2-9   epilogue (both CTAs): warp w reads TMEM lanes 32*(w%4).. and one 128-column
//               half of the tile, keeps 128 running sums per thread, stores once per tile.
#include "tc_common.cuh"

namespace gemm_gb300 {
namespace {

using namespace tc;

constexpr int kXThreads = 320;
constexpr int kXEpiWarps = 8;

template <bool F16ACC>
struct CfgX {
  static constexpr int ES = F16ACC ? 2 : 4;     // bytes per operand element
  static constexpr int BM = kTcBlockM;          // rows per CTA (256 per pair)
  static constexpr int BN = 256;                // columns per pair tile
  static constexpr int BN_HALF = BN / 2;        // B columns loaded by each CTA
  static constexpr int BK = kRowBytes / ES;     // elements per 128-byte K-block
  static constexpr int UMMA_K = F16ACC ? 16 : 8;  // K per tcgen05.mma (kind::f16 / kind::tf32)
  static constexpr int K_STEPS = BK / UMMA_K;
  static constexpr int A_BYTES = BM * kRowBytes;
  static constexpr int B_BYTES = BN_HALF * kRowBytes;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr int STAGES = 6;
  static constexpr int EPI_OFFSET = STAGES * STAGE_BYTES;
  static constexpr int EPI_BYTES = kXEpiWarps * kStoreBufBytes;  // one staging box per warp
  static constexpr int BAR_OFFSET = EPI_OFFSET + EPI_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 5;
  // + TMEM address, abort flag and the four teardown words (see `xs` in the kernel)
  static constexpr int SMEM_BYTES = BAR_OFFSET + NUM_BARS * 8 + 32 + 1024;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr int COLS = 128;  // columns per epilogue thread
  static_assert(K_STEPS == 4, "four MMAs per K-block");
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};
constexpr int kXCols = 128;

// Store one warp's 32 x 128 block from registers through the 128B-swizzled staging box.
template <int OUT>
__device__ __forceinline__ void store_regs_tma(const float (&v)[kXCols], const CUtensorMap *tmC,
                                               uint8_t *sb, int lane, int row0, int col0, int M,
                                               int N) {
  constexpr int OUT_COLS = OUT == GEMM_F32 ? 32 : 64;
  if (row0 >= M) return;  // warp-uniform
#pragma unroll
  for (int b = 0; b < kXCols / OUT_COLS; ++b) {
    if (col0 + b * OUT_COLS >= N) break;  // warp-uniform
    if (lane == 0) bulk_wait_group_read<0>();
    __syncwarp();
    const uint32_t row_addr = smem_u32(sb) + lane * kRowBytes;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      uint32_t w0, w1, w2, w3;
      if (OUT == GEMM_F32) {
        const int c = b * 32 + ch * 4;
        w0 = __float_as_uint(v[c]), w1 = __float_as_uint(v[c + 1]);
        w2 = __float_as_uint(v[c + 2]), w3 = __float_as_uint(v[c + 3]);
      } else {
        const int c = b * 64 + ch * 8;
        w0 = pack2<OUT>(__float_as_uint(v[c]), __float_as_uint(v[c + 1]));
        w1 = pack2<OUT>(__float_as_uint(v[c + 2]), __float_as_uint(v[c + 3]));
        w2 = pack2<OUT>(__float_as_uint(v[c + 4]), __float_as_uint(v[c + 5]));
        w3 = pack2<OUT>(__float_as_uint(v[c + 6]), __float_as_uint(v[c + 7]));
      }
      const uint32_t dst = row_addr + ((ch ^ (lane & 7)) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(dst), "r"(w0), "r"(w1),
                   "r"(w2), "r"(w3)
                   : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmC, smem_u32(sb), col0 + b * OUT_COLS, row0);
      bulk_commit_group();
    }
  }
}

// Store one thread's row segment from registers with plain masked stores.
template <int OUT>
__device__ __forceinline__ void store_regs_direct(const float (&v)[kXCols], const TcParams &p,
                                                  int row, int col0) {
  if (row >= p.M || col0 >= p.N) return;
  const int n = min(kXCols, p.N - col0);
  const int64_t base = static_cast<int64_t>(row) * p.ldc + col0;
#pragma unroll
  for (int j = 0; j < kXCols; ++j) {
    if (j < n) {
      if (OUT == GEMM_F32)
        reinterpret_cast<float *>(p.C)[base + j] = v[j];
      else if (OUT == GEMM_BF16)
        reinterpret_cast<__nv_bfloat16 *>(p.C)[base + j] = __float2bfloat16_rn(v[j]);
      else
        reinterpret_cast<__half *>(p.C)[base + j] = __float2half_rn(v[j]);
    }
  }
}

template <int OUT>
__device__ __forceinline__ void store_regs(const float (&v)[kXCols], const CUtensorMap *tmC,
                                           uint8_t *sb, const TcParams &p, int lane, int row0,
                                           int col0) {
  if (p.tma_store)
    store_regs_tma<OUT>(v, tmC, sb, lane, row0, col0, p.M, p.N);
  else
    store_regs_direct<OUT>(v, p, row0 + lane, col0);
}

template <bool F16ACC>
__global__ void __launch_bounds__(kXThreads, 1)
    tc_chunk_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmP,
                    const TcParams p) {
  using G = CfgX<F16ACC>;
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
  // Teardown words, as in the CTA-pair kernel: [0] stage fills this CTA's loader issued,
  // [1] fills the MMA issuer consumed (leader), [2] the peer's issued fills (written by the
  // peer into the leader), [3] whether the other CTA aborted.
  volatile uint32_t *xs = reinterpret_cast<volatile uint32_t *>(tmem_slot + 2);

  const int warp = threadIdx.x / 32;
  const int lane = threadIdx.x % 32;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int chunk = p.chunk_steps;  // MMA instructions per TMEM partial

  if (threadIdx.x == 0) {
    for (int s = 0; s < G::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tmem_full[b], 1);
      mbar_init(&tmem_empty[b], 2 * kXEpiWarps);  // every epilogue warp of both CTAs
    }
    mbar_init(drain, 1);
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
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // The prologue above may overlap the previous kernel on the stream (the operand split
  // copies, in exact mode); global memory only from here on.
  grid_dependency_wait();
  grid_launch_dependents();
  const Watchdog wd{abort_flag, p.status, p.timeout_ns};
  const int cluster_id = blockIdx.x / 2;
  const int num_clusters = gridDim.x / 2;
  // Whole tiles round-robin over the clusters, then (exact mode) the split-K share.
  const SkSchedule sched = sk_make(p.tiles_m * p.tiles_n, p.k_blocks, num_clusters, p.sk_dp_tiles);
  const bool split = p.sk_dp_tiles < p.tiles_m * p.tiles_n;
  const int epoch = split ? sk_epoch_begin(p.sk_epoch_word) : 0;
  // Chunks are whole K-blocks in exact mode (the issuer then decides once per K-block);
  // the fp16 accumulator may round every one or few MMAs.
  const bool by_block = chunk % G::K_STEPS == 0;
  const int chunk_kb = by_block ? chunk / G::K_STEPS : 1;
  auto chunks_of = [&](const SkSegment &seg) {
    const int len = seg.kb_end - seg.kb_begin;
    return by_block ? (len + chunk_kb - 1) / chunk_kb : (len * G::K_STEPS + chunk - 1) / chunk;
  };

  if (warp == 0) {
    // ------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, issued = 0;
      bool ok = (p.debug_flags & kDebugStallProducer) == 0;
      const int stop_after = stall_after_fills(p.debug_flags, static_cast<int>(rank));
      const uint64_t keep = l2_policy_evict_last();  // operand tiles stay in L2 longest
      WorkIter work(sched, cluster_id);
      SkSegment seg;
      while (ok && work.next(seg)) {
        int pm, pn;
        tile_coords(seg.tile, p.tiles_m, p.tiles_n, p.group_m, pm, pn);
        const int m0 = pm * (2 * G::BM) + static_cast<int>(rank) * G::BM;
        const int n0 = pn * G::BN + static_cast<int>(rank) * G::BN_HALF;
        for (int kb = seg.kb_begin; kb < seg.kb_end; ++kb) {
          if (stop_after >= 0 && issued >= static_cast<uint32_t>(stop_after)) {
            ok = false;  // test hook: this loader stops here, copies still in flight
            break;
          }
          if (!mbar_wait_cluster(&empty[stage], phase ^ 1, wd)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * G::STAGE_BYTES);
          const uint32_t a_dst = smem_u32(smem + stage * G::STAGE_BYTES);
          const uint32_t fb = mapa_shared(smem_u32(&full[stage]), 0);
          int xa = kb * G::BK, xb = xa;  // K coordinates of the A and B boxes
          if (!F16ACC) {
            // K-block j of product q reads A's part (q == 2 ? lo : hi), B's (q == 1 ? lo : hi)
            const int q = kb / p.split_kb, j = kb - q * p.split_kb;
            xa = (j + (q == 2 ? p.split_kb : 0)) * G::BK;
            xb = (j + (q == 1 ? p.split_kb : 0)) * G::BK;
          }
          tma_load_2d_pair_hint(a_dst, &tmA, fb, xa, m0, keep);
          tma_load_2d_pair_hint(a_dst + G::A_BYTES, &tmB, fb, xb, n0, keep);
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
      // Four MMAs per K-block. When chunks are whole K-blocks (always in exact mode) the
      // chunk decisions are taken once per K-block and the four MMAs issue back to back:
      // this single thread's issue rate bounds the kernel, and per-MMA branching was
      // measured to cost up to half of the throughput. Chunks start at each piece's first
      // K-block.
      auto take_acc = [&](uint32_t &d_tmem) {  // a fresh accumulator for the next chunk
        if (!mbar_wait_cluster(&tmem_empty[acc], acc_phase ^ 1, wd)) return false;
        tc_fence_after();
        d_tmem = tmem_base + acc * G::BN;
        return true;
      };
      auto hand_over = [&]() {  // chunk done: the epilogue may read it
        mma_commit_pair_multicast(&tmem_full[acc], 0x3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      };
      WorkIter work(sched, cluster_id);
      SkSegment seg;
      auto next_stage = [&]() {
        if (++stage == G::STAGES) {
          stage = 0;
          phase ^= 1;
        }
      };
      while (ok && work.next(seg)) {
        uint32_t d_tmem = 0;
        if (by_block) {
          // chunk by chunk: a fresh accumulator, then a tight loop over its K-blocks
          for (int c0 = seg.kb_begin; ok && c0 < seg.kb_end; c0 += chunk_kb) {
            if (!take_acc(d_tmem)) {
              ok = false;
              break;
            }
            const int c1 = c0 + chunk_kb < seg.kb_end ? c0 + chunk_kb : seg.kb_end;
            for (int kb = c0; kb < c1; ++kb) {
              if (!mbar_wait_cluster(&full[stage], phase, wd)) {
                ok = false;
                break;
              }
              ++consumed;
              tc_fence_after();
              const uint32_t a_base = smem_u32(smem + stage * G::STAGE_BYTES);
              const uint32_t b_base = a_base + G::A_BYTES;
#pragma unroll
              for (int kk = 0; kk < G::K_STEPS; ++kk) {
                const uint64_t ad = sdesc_sw128(a_base + kk * 32, 16, 1024);
                const uint64_t bd = sdesc_sw128(b_base + kk * 32, 16, 1024);
                const uint32_t accumulate = (kb != c0) || kk != 0;
                if (F16ACC)
                  mma_f16_pair(d_tmem, ad, bd, p.idesc, accumulate);
                else
                  mma_tf32_pair(d_tmem, ad, bd, p.idesc, accumulate);
              }
              mma_commit_pair_multicast(&empty[stage], 0x3);
              next_stage();
            }
            if (!ok) break;
            hand_over();
          }
          continue;
        }
        int left = 0;  // MMAs left in the current chunk (0: start one)
        for (int kb = seg.kb_begin; ok && kb < seg.kb_end; ++kb) {
          if (!mbar_wait_cluster(&full[stage], phase, wd)) {
            ok = false;
            break;
          }
          ++consumed;
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + stage * G::STAGE_BYTES);
          const uint32_t b_base = a_base + G::A_BYTES;
          const bool last_kb = kb == seg.kb_end - 1;
#pragma unroll
          for (int kk = 0; kk < G::K_STEPS; ++kk) {
            const bool fresh = left == 0;
            if (fresh) {
              if (!take_acc(d_tmem)) {
                ok = false;
                break;
              }
              left = chunk;
            }
            const uint64_t ad = sdesc_sw128(a_base + kk * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(b_base + kk * 32, 16, 1024);
            if (F16ACC)
              mma_f16_pair(d_tmem, ad, bd, p.idesc, fresh ? 0u : 1u);
            else
              mma_tf32_pair(d_tmem, ad, bd, p.idesc, fresh ? 0u : 1u);
            if (--left == 0 || (last_kb && kk == G::K_STEPS - 1)) {
              hand_over();
              left = 0;
            }
          }
          mma_commit_pair_multicast(&empty[stage], 0x3);
          next_stage();
        }
      }
      mma_commit_pair(drain);
      drain_wait(drain, 0, p.timeout_ns);
      xs[1] = consumed;
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------ epilogue (both CTAs)
    const int e = warp - 2;
    const int quarter = warp & 3;
    const int half = e >> 2;  // which 128 columns of the tile
    uint8_t *sb = smem + G::EPI_OFFSET + e * kStoreBufBytes;
    uint32_t acc = 0, acc_phase = 0;
    bool ok = true;
    WorkIter work(sched, cluster_id);
    SkSegment seg;
    while (ok && work.next(seg)) {
      const int chunks = chunks_of(seg);
      // The tile's running sums start at zero once: fp32 values (exact mode) or fp16 pairs
      // (fp16 accumulator; +0 is the all-zero bit pattern).
      float sum[F16ACC ? 1 : G::COLS];
      __half2 hsum[F16ACC ? G::COLS / 2 : 1];
      if (F16ACC) {
#pragma unroll
        for (int j = 0; j < G::COLS / 2; ++j) hsum[j] = __floats2half2_rn(0.0f, 0.0f);
      } else {
#pragma unroll
        for (int j = 0; j < G::COLS; ++j) sum[j] = 0.0f;
      }
      for (int c = 0; c < chunks; ++c) {
        bool got = mbar_wait_cluster_inline(&tmem_full[acc], acc_phase, wd);
        got = __all_sync(0xffffffffu, got);
        if (!got) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t t = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                           acc * G::BN + half * G::COLS;
#pragma unroll
        if (F16ACC) {
          // two 32-column reads in flight per wait (the chunk's drain is this kernel's
          // critical path when chunks are single MMAs); partial = fp16(chunk dot),
          // acc = fp16(acc + partial)
#pragma unroll
          for (int q = 0; q < G::COLS / 32; q += 2) {
            uint32_t r[2][32];
            tmem_ld_32x32b_x32(t + q * 32, r[0]);
            tmem_ld_32x32b_x32(t + (q + 1) * 32, r[1]);
            tmem_wait_ld();
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
              for (int j = 0; j < 16; ++j)
                hsum[(q + h2) * 16 + j] =
                    __hadd2(hsum[(q + h2) * 16 + j],
                            __floats2half2_rn(__uint_as_float(r[h2][2 * j]),
                                              __uint_as_float(r[h2][2 * j + 1])));
          }
        } else {
#pragma unroll
          for (int q = 0; q < G::COLS / 32; ++q) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(t + q * 32, r);
            tmem_wait_ld();
#pragma unroll
            for (int j = 0; j < 32; ++j) sum[q * 32 + j] += __uint_as_float(r[j]);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(mapa_shared(smem_u32(&tmem_empty[acc]), 0));
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1;
      }
      if (!ok) break;
      // Split-K pieces (exact mode only): this warp's 32 x 128 block of the tile lives at
      // rows (worker * 2 + rank) * 128 + quarter * 32 of the workspace, columns half * 128.
      const int part_row = quarter * 32;
      int *const flags = p.sk_flags;
      if constexpr (!F16ACC) {
      if (seg.role == kSegPartial) {
        store_regs_tma<GEMM_F32>(sum, &tmP, sb, lane, (cluster_id * 2 + rank) * G::BM + part_row,
                                 half * G::COLS, INT32_MAX, G::BN);
        if (lane == 0) {
          bulk_wait_group<0>();  // the partial's writes are complete
          fence_proxy_async_global();
          st_release_gpu(flags + (cluster_id * 2 + rank) * kXEpiWarps + e, epoch);
        }
        __syncwarp();
        goto next_segment;
      }
      if (seg.role == kSegOwner) {
        // add the partials of the workers that computed the start of this tile, lowest first
        for (int w = seg.first_src; ok && w <= seg.last_src; ++w) {
          ok = wait_flag(flags + (w * 2 + rank) * kXEpiWarps + e, epoch, wd);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
          const float4 *src = reinterpret_cast<const float4 *>(
              p.sk_partials + (static_cast<int64_t>((w * 2 + rank) * G::BM + part_row + lane)) *
                                  G::BN + half * G::COLS);
#pragma unroll
          for (int j = 0; j < G::COLS / 4; ++j) {
            const float4 v = src[j];
            sum[4 * j] += v.x, sum[4 * j + 1] += v.y, sum[4 * j + 2] += v.z, sum[4 * j + 3] += v.w;
          }
        }
        if (!ok) break;
      }
      }
      {
      int pm, pn;
      tile_coords(seg.tile, p.tiles_m, p.tiles_n, p.group_m, pm, pn);
      const int row0 = pm * (2 * G::BM) + static_cast<int>(rank) * G::BM + quarter * 32;
      const int col0 = pn * G::BN + half * G::COLS;
      float out[kXCols];
#pragma unroll
      for (int j = 0; j < kXCols; ++j)
        out[j] = F16ACC ? (j % 2 ? __high2float(hsum[j / 2]) : __low2float(hsum[j / 2])) : sum[j];
      if (p.out_dtype == GEMM_BF16)
        store_regs<GEMM_BF16>(out, &tmC, sb, p, lane, row0, col0);
      else if (p.out_dtype == GEMM_F16)
        store_regs<GEMM_F16>(out, &tmC, sb, p, lane, row0, col0);
      else
        store_regs<GEMM_F32>(out, &tmC, sb, p, lane, row0, col0);
      }
    next_segment:;
    }
    if (lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  __syncthreads();
  // As in the CTA-pair kernel: exchange abort states; after an abort the leader accounts
  // for and waits for every stage fill either CTA's loader issued before either leaves.
  if (threadIdx.x == 0) {
    st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t *>(&xs[3])), rank ^ 1u),
                          *abort_flag ? 1u : 0u);
    if (!leader) st_shared_cluster_u32(mapa_shared(smem_u32(const_cast<uint32_t *>(&xs[2])), 0), xs[0]);
  }
  tc_fence_before();
  cluster_sync();
  if (*abort_flag || xs[3]) {
    if (leader && threadIdx.x == 0)
      drain_pair_fills<G::STAGES>(full, xs[1], xs[0], xs[2], G::STAGE_BYTES, p.timeout_ns);
    cluster_sync();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, G::TMEM_COLS);
  }
  if (split && threadIdx.x == 0) sk_epoch_end(p.sk_epoch_word, epoch);
}

template <bool F16ACC>
cudaLaunchConfig_t chunk_config(int grid, cudaStream_t s, cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kXThreads, 1, 1);
  cfg.dynamicSmemBytes = CfgX<F16ACC>::SMEM_BYTES;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <bool F16ACC>
int max_active_clusters() {
  static int cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  if (cached[dev] > 0) return cached[dev];
  if (cudaFuncSetAttribute(tc_chunk_kernel<F16ACC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           CfgX<F16ACC>::SMEM_BYTES) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = chunk_config<F16ACC>(2, nullptr, attr);
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_chunk_kernel<F16ACC>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cached[dev] = n;
  return n;
}

template <bool F16ACC>
cudaError_t launch(const CUtensorMap &tmA, const CUtensorMap &tmB, const CUtensorMap &tmC,
                   const CUtensorMap &tmP, const TcParams &p, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(
      tc_chunk_kernel<F16ACC>, cudaFuncAttributeMaxDynamicSharedMemorySize, CfgX<F16ACC>::SMEM_BYTES);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = chunk_config<F16ACC>(grid, s, attr);
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see grid_dependency_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tc_chunk_kernel<F16ACC>, tmA, tmB, tmC, tmP, p);
}

}  // namespace

int tc_chunk_max_active_clusters(bool f16acc) {
  return f16acc ? max_active_clusters<true>() : max_active_clusters<false>();
}

cudaError_t tc_chunk_launch(bool f16acc, const CUtensorMap &tmA, const CUtensorMap &tmB,
                            const CUtensorMap &tmC, const CUtensorMap &tmP, const TcParams &p,
                            int grid, cudaStream_t s) {
  return f16acc ? launch<true>(tmA, tmB, tmC, tmP, p, grid, s)
                : launch<false>(tmA, tmB, tmC, tmP, p, grid, s);
}

}  // namespace gemm_gb300
