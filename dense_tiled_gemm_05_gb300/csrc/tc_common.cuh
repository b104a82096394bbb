// tc_common.cuh -- pieces shared by the single-CTA and CTA-pair tensor-core kernels:
// the grouped tile raster, the teardown wait, and the two epilogue forms (TMA store
// through a 128B-swizzled staging box, or plain masked stores).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"
#include "sk_schedule.h"

namespace gemm_gb300 {
namespace tc {

constexpr int kThreads = 192;  // warp 0 producer, warp 1 MMA, warps 2-5 epilogue
constexpr int kEpiWarps = 4;
constexpr int kRowBytes = 128;                   // one 128-byte swizzle row
constexpr int kStoreBufBytes = 32 * kRowBytes;   // one epilogue staging box: 32 rows x 128 B

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
static __device__ __noinline__ void drain_wait(uint64_t *bar, uint32_t parity, uint64_t timeout_ns) {
  const uint32_t a = smem_u32(bar);
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(a, parity)) {
    if (global_timer_ns() - t0 > timeout_ns) return;
  }
}

// Teardown of a CTA pair after an abort. Both CTAs' TMA loads signal the leader's full
// barriers: a stage fill is complete when the leader's producer has arrived (expecting the
// bytes of both CTAs) and both CTAs' bytes have landed. Fills numbered `consumed` and on
// (the MMA issuer waited for all earlier ones) may still be in flight: the leader issued
// `leader_issued` fills, the peer `peer_issued`, and the two differ when one producer
// stopped first. For each outstanding fill the leader completes the barrier's accounting
// for the side that never issued it -- the peer's bytes it still expects, or the arrival
// and the peer's bytes when only the peer issued -- and waits (bounded) for the phase, so
// every copy either CTA issued has landed when this returns. At most STAGES fills are
// outstanding (a producer reuses a stage only after the MMAs have consumed it), so each
// stage has at most one outstanding phase.
template <int STAGES>
__device__ __noinline__ void drain_pair_fills(uint64_t *full, uint32_t consumed,
                                              uint32_t leader_issued, uint32_t peer_issued,
                                              uint32_t peer_bytes, uint64_t timeout_ns) {
  const uint32_t end = leader_issued > peer_issued ? leader_issued : peer_issued;
  for (uint32_t i = consumed; i < end; ++i) {
    uint64_t *bar = &full[i % STAGES];
    if (i >= leader_issued)
      mbar_arrive_expect_tx(bar, peer_bytes);  // only the peer issued this fill
    else if (i >= peer_issued)
      mbar_complete_tx(bar, peer_bytes);  // the peer's part of this fill never comes
    drain_wait(bar, (i / STAGES) & 1, timeout_ns);
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

// Epilogue, direct form for a C that TMA cannot address (misaligned base or ldc), and for
// the warp a shortened tile ends in: each lane owns one row and writes its in-range
// columns with plain stores (a lane given a row at or past M stores nothing).
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

// Split-K owner: adds one partial (this warp's 32 rows x BN fp32, already TMA-loaded into
// `slice` as BN/32 128B-swizzled boxes of 32 rows x 32 columns) into its TMEM rows.
template <int BN>
__device__ __forceinline__ void add_partial_into_tmem(uint32_t t_row, const uint8_t *slice,
                                                      int lane) {
#pragma unroll 1
  for (int c0 = 0; c0 < BN; c0 += 32) {
    uint32_t r[32];
    tmem_ld_32x32b_x32(t_row + c0, r);
    tmem_wait_ld();
    const uint32_t row_addr = smem_u32(slice + (c0 / 32) * kStoreBufBytes) + lane * kRowBytes;
#pragma unroll
    for (int ch = 0; ch < 8; ++ch) {
      float4 v;
      asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                   : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                   : "r"(row_addr + ((ch ^ (lane & 7)) << 4)));
      r[4 * ch + 0] = __float_as_uint(__uint_as_float(r[4 * ch + 0]) + v.x);
      r[4 * ch + 1] = __float_as_uint(__uint_as_float(r[4 * ch + 1]) + v.y);
      r[4 * ch + 2] = __float_as_uint(__uint_as_float(r[4 * ch + 2]) + v.z);
      r[4 * ch + 3] = __float_as_uint(__uint_as_float(r[4 * ch + 3]) + v.w);
    }
    tmem_st_32x32b_x32(t_row + c0, r);
  }
  tmem_wait_st();
}

__device__ __forceinline__ void st_release_gpu(int *p, int v) {
  asm volatile("st.release.gpu.global.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ int ld_acquire_gpu(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Split-K epochs. A partial writer stores `epoch` in its flag; the owner waits for that
// value. Every CTA of a launch reads the epoch word once at its start (it is stable then:
// only the last CTA of the previous launch changed it) and uses epoch = word + 1; the last
// CTA of the launch to finish stores that epoch into the word. Flags left by an earlier
// launch -- also one that gave up on a bounded wait, or a replayed graph -- hold an older
// value and never match.
__device__ __forceinline__ int sk_epoch_begin(const int *word) {
  return *reinterpret_cast<const volatile int *>(word) + 1;
}
__device__ __forceinline__ void sk_epoch_end(int *word, int epoch) {
  __threadfence();
  if (atomicAdd(word + 1, 1) == static_cast<int>(gridDim.x) - 1) {
    word[1] = 0;
    *reinterpret_cast<volatile int *>(word) = epoch;
  }
}

// Bounded wait until *flag == value (a split-K partial of this launch is in memory).
__device__ __forceinline__ bool wait_flag(const int *flag, int value, const Watchdog &wd) {
  if (ld_acquire_gpu(flag) == value) return true;
  const uint64_t t0 = global_timer_ns();
  while (ld_acquire_gpu(flag) != value) {
    if (*wd.abort_flag) return false;
    if (global_timer_ns() - t0 > wd.timeout_ns) {
      atomicCAS(wd.status, 0, kStatusTimeout);
      *wd.abort_flag = 1;
      __threadfence_block();
      return false;
    }
    __nanosleep(64);
  }
  return true;
}

// The pieces of work of one persistent worker: its round-robin whole tiles, then its
// split-K share (see sk_schedule.h). Every role of a worker walks the same sequence.
struct WorkIter {
  SkSchedule S;
  int32_t slot, dp_i, dp_n;
  int64_t lo, hi;  // split-K units still to do: [lo, hi)
  __device__ __forceinline__ WorkIter(const SkSchedule &s, int32_t w) : S(s), slot(w), dp_i(0) {
    dp_n = sk_dp_count(S, slot);
    lo = sk_begin(S, slot);
    hi = sk_begin(S, slot + 1);
  }
  __device__ __forceinline__ bool next(SkSegment &seg) {
    if (dp_i < dp_n) {
      seg.tile = slot + dp_i * S.slots;
      seg.kb_begin = 0;
      seg.kb_end = S.kb;
      seg.role = kSegFull;
      seg.first_src = seg.last_src = -1;
      ++dp_i;
      return true;
    }
    if (hi > lo) {  // the split-K share, walked from its end to its start
      hi = sk_segment_at(S, slot, hi, &seg);
      return true;
    }
    return false;
  }
};

}  // namespace tc
}  // namespace gemm_gb300
