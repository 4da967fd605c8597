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

}  // namespace csa2
