// sk_schedule.h -- how a persistent grid of `slots` workers (CTA clusters) divides the
// output tiles of one product when their number does not fill whole rounds.
//
// Each output tile is the K-loop of "Chapter 13: The Blocked Matmul Kernel", section 13.1:
// `kb` K-blocks whose partial products are summed into one accumulator. The first
// `dp_tiles` tiles go round-robin to the slots whole ("data-parallel" rounds). The
// remaining tiles are cut into their (tile, K-block) units, and every slot takes one
// contiguous, equal share of those units ("stream-K"), so the last round ends at the same
// time on every slot. A slot walks its share from the end to the start, in segments of at
// most one tile: a segment covering a whole tile is stored as usual; a segment that lacks
// its tile's last K-block is a *partial*: its fp32 sum goes to the slot's workspace entry;
// the segment that holds a tile's last K-block but not all of it is the tile's *owner*: it
// adds the partials of the slots that cover the start of that tile, in increasing slot
// order, and stores the result. Walking backwards makes a slot's partial its first
// segment (written early) and its owner segment its last (waiting late), and an owner only
// ever waits for slots with smaller numbers, which the GPU dispatches no later than the
// owner itself: the waits cannot block each other. Every slot has at most one partial
// segment, so workspace entries are indexed by slot.
//
// Pure integer arithmetic, shared by the host planner and the device kernels.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define SK_HD __host__ __device__ __forceinline__
#else
#define SK_HD inline
#endif

namespace gemm_gb300 {

enum : int32_t { kSegFull = 0, kSegPartial = 1, kSegOwner = 2 };

struct SkSchedule {
  int32_t tiles;     // output tiles
  int32_t kb;        // K-blocks per tile
  int32_t slots;     // workers
  int32_t dp_tiles;  // tiles done whole, round-robin (a multiple of slots, or all tiles)
  // derived
  int64_t sk_units;  // (tiles - dp_tiles) * kb
};

struct SkSegment {
  int32_t tile;       // output tile index
  int32_t kb_begin;   // first K-block
  int32_t kb_end;     // one past the last K-block
  int32_t role;       // kSegFull, kSegPartial or kSegOwner
  int32_t first_src;  // owner: first slot whose partial it adds (all lower than the owner)
  int32_t last_src;   // owner: last slot whose partial it adds
};

// Units [sk_begin(s), sk_begin(s+1)) belong to slot s.
SK_HD int64_t sk_begin(const SkSchedule &S, int64_t s) { return s * S.sk_units / S.slots; }

// The slot whose share holds stream-K unit u (0 <= u < sk_units).
SK_HD int32_t sk_slot_of_unit(const SkSchedule &S, int64_t u) {
  // the largest s with floor(s * U / slots) <= u
  int64_t s = ((u + 1) * S.slots - 1) / S.sk_units;
  if (s >= S.slots) s = S.slots - 1;
  while (s > 0 && sk_begin(S, s) > u) --s;
  while (s + 1 < S.slots && sk_begin(S, s + 1) <= u) ++s;
  return static_cast<int32_t>(s);
}

SK_HD SkSchedule sk_make(int32_t tiles, int32_t kb, int32_t slots, int32_t dp_tiles) {
  SkSchedule S;
  S.tiles = tiles;
  S.kb = kb;
  S.slots = slots;
  S.dp_tiles = dp_tiles;
  S.sk_units = static_cast<int64_t>(tiles - dp_tiles) * kb;
  return S;
}

// Whole tiles done round-robin: all of them when they fill whole rounds, when stream-K is
// off, or when the split units would not give every slot at least one; otherwise all but
// the last full round and the partial round, which go stream-K. With every share
// non-empty, the slots after an owner up to the one finishing its tile all start inside
// that tile, i.e. are exactly its partial writers.
SK_HD int32_t sk_dp_tiles(int32_t tiles, int32_t kb, int32_t slots, bool stream_k) {
  if (!stream_k || slots <= 1 || tiles % slots == 0) return tiles;
  const int32_t full = tiles / slots;
  const int32_t dp = full > 0 ? (full - 1) * slots : 0;
  if (static_cast<int64_t>(tiles - dp) * kb < slots) return tiles;
  return dp;
}

// Number of whole tiles slot s does round-robin.
SK_HD int32_t sk_dp_count(const SkSchedule &S, int32_t s) {
  return S.dp_tiles / S.slots + (s < S.dp_tiles % S.slots ? 1 : 0);
}

// The stream-K segment of slot s that ends at unit u (exclusive; inside s's share, walking
// backwards from the share's end); returns the unit where it starts, i.e. where the slot's
// next segment ends.
SK_HD int64_t sk_segment_at(const SkSchedule &S, int32_t s, int64_t u, SkSegment *seg) {
  const int64_t lo = sk_begin(S, s);
  const int64_t t = (u - 1) / S.kb;  // stream-K tile number
  const int64_t begin = t * S.kb > lo ? t * S.kb : lo;
  seg->tile = static_cast<int32_t>(S.dp_tiles + t);
  seg->kb_begin = static_cast<int32_t>(begin - t * S.kb);
  seg->kb_end = static_cast<int32_t>(u - t * S.kb);
  seg->first_src = seg->last_src = -1;
  if (seg->kb_end < S.kb) {
    seg->role = kSegPartial;
  } else if (seg->kb_begin > 0) {
    seg->role = kSegOwner;
    seg->first_src = sk_slot_of_unit(S, t * S.kb);
    seg->last_src = s - 1;
  } else {
    seg->role = kSegFull;
  }
  return begin;
}

}  // namespace gemm_gb300
