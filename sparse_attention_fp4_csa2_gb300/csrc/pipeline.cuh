// Bookkeeping of the persistent, warp-specialised sweeps: the slot and phase
// of an mbarrier-guarded ring, and the (sequence, tile) a CTA works on, both
// advanced per tile without division (each role's loop runs on one thread,
// where a 64-bit division per tile costs hundreds of cycles).
#pragma once
#include "kernels.cuh"

namespace csa2 {

template <int N>
struct Ring {
  int slot = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next() {
    if (++slot == N) {
      slot = 0;
      phase ^= 1u;
    }
  }
};

struct TileCursor {
  int b, t, per_seq;
  __device__ __forceinline__ TileCursor(int64_t it, int tiles_per_seq)
      : b((int)(it / tiles_per_seq)), t((int)(it % tiles_per_seq)), per_seq(tiles_per_seq) {}
  __device__ __forceinline__ void next() {
    if (++t == per_seq) {
      t = 0;
      ++b;
    }
  }
};

// Lane 0's value for the whole warp when the warp runs the loop together
// (pool tiles); the value itself when lane 0 runs it alone (Full tiles).
template <bool kWarp>
__device__ __forceinline__ int warp_bcast(int v) {
  if constexpr (kWarp) return __shfl_sync(0xffffffffu, v, 0);
  return v;
}

// ------------------------------------------------ row histograms of a sweep
// The sweeps count every score's top-K key for the cluster top-K of the same
// call (TOPK_HIST_BITS bins per row).  In shared memory: two slots of
// TOPK_HIST_BINS 16-bit counts, two bins to a word, used by segments of a
// CTA's tiles -- the tiles of one row, at most a segment's tile limit, so
// that no count passes 65,535 -- by segment parity.
constexpr int kHistWords = TOPK_HIST_BINS / 2;   // words per slot

__device__ __forceinline__ void hist_count(uint32_t *slot, float score) {
  const uint32_t key = topk_score_key(score);
  if (key) {
    const uint32_t bin = key >> (32 - TOPK_HIST_BITS);
    atomicAdd(slot + (bin >> 1), (bin & 1u) ? 0x10000u : 1u);
  }
}

// The four epilogue warps' walk over the segments (each warp its own copy,
// quadrant `quad` of 0..3; every warp sees the same tiles in the same order).
// At a segment's end the four warps meet on hseg[slot]; each adds its quarter
// of the slot into the row's global histogram and clears it, then arrives on
// hfree[slot], which the segment two later awaits before adding to the slot.
// A warp runs at most one tile ahead of the others (the accumulator ring),
// so two slots suffice.  Waits are bounded (mbar_wait).
struct HistSegments {
  uint64_t *hseg, *hfree;
  uint32_t *slots, *global;
  int seg_tiles, quad, lane;
  int seg = -1, left = 0, row = -1;

  __device__ __forceinline__ HistSegments(uint64_t *hs, uint64_t *hf, uint32_t *sl, uint32_t *g, int st, int q, int l)
      : hseg(hs), hfree(hf), slots(sl), global(g), seg_tiles(st), quad(q), lane(l) {}

  // Before tile (row b): a new segment at a row change or after seg_tiles tiles.
  __device__ __forceinline__ void tile(int b) {
    if (!global) return;
    if (b != row || left == 0) {
      end();
      ++seg;
      left = seg_tiles;
      row = b;
      if (seg >= 2) mbar_wait(&hfree[seg & 1], (uint32_t)((seg >> 1) - 1) & 1u);
    }
    --left;
  }
  // The current segment's slot, or NULL when no histogram is kept.
  __device__ __forceinline__ uint32_t *slot() const { return global ? slots + (seg & 1) * kHistWords : nullptr; }
  // After the last tile.
  __device__ __forceinline__ void finish() {
    if (global) end();
  }

 private:
  __device__ __forceinline__ void end() {
    if (seg < 0) return;
    const int p = seg & 1;
    __syncwarp();
    if (lane == 0) mbar_arrive(&hseg[p]);
    mbar_wait(&hseg[p], (uint32_t)(seg >> 1) & 1u);
    uint32_t *hs = slots + p * kHistWords;
    uint32_t *g = global + (int64_t)row * TOPK_HIST_BINS;
    constexpr int kQuarter = kHistWords / 4;
#pragma unroll 4
    for (int i = quad * kQuarter + lane; i < (quad + 1) * kQuarter; i += 32) {
      const uint32_t c = hs[i];
      if (c) {
        hs[i] = 0u;
        if (c & 0xFFFFu) atomicAdd(g + 2 * i, c & 0xFFFFu);
        if (c >> 16) atomicAdd(g + 2 * i + 1, c >> 16);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&hfree[p]);
  }
};

}  // namespace csa2
