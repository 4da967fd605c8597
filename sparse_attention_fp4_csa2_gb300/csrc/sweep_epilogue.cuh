// Epilogue of the indexer sweeps (bf16 and MXFP4): one tile row's score from
// its 32 head dot products, and the HSI block score of its block of 8.
#pragma once
#include "kernels.cuh"

namespace csa2 {

// Row r of tile t of sequence b: score = sum_h w_h ReLU(dot_h) ("DeepSeek-
// V4.1-Flash - Architecture", section 2), -inf where the position is not
// visible; the Full sweep also writes the max (or sum) over each block of 8
// ("DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression", 2.3.4).
// Called by all 32 lanes of a warp (the block reduction shuffles).
template <bool kPool>
__device__ __forceinline__ void sweep_store_row(const SweepArgs &a, int b, int t, int r, int lane, int32_t nv,
                                                const float (&wv)[HI], const uint32_t (&v)[32]) {
  float sc = 0.0f;
#pragma unroll
  for (int h = 0; h < HI; ++h) sc = fmaf(wv[h], fmaxf(__uint_as_float(v[h]), 0.0f), sc);
  float *srow = a.scores + (int64_t)b * a.row_len;
  if (!kPool) {
    const int64_t pos = (int64_t)t * SWEEP_TILE + r;
    const bool valid = pos < nv;
    srow[pos] = valid ? sc : -INFINITY;
    if (a.block_scores) {
      float bv;
      if (a.block_reduce == 0) {
        bv = valid ? sc : -INFINITY;
        bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, 1));
        bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, 2));
        bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, 4));
      } else {
        bv = valid ? sc : 0.0f;
        bv += __shfl_xor_sync(0xffffffffu, bv, 1);
        bv += __shfl_xor_sync(0xffffffffu, bv, 2);
        bv += __shfl_xor_sync(0xffffffffu, bv, 4);
        if ((pos & ~int64_t(BLOCK - 1)) >= nv) bv = -INFINITY;
      }
      const int64_t blk = pos / BLOCK;
      if ((lane & (BLOCK - 1)) == 0 && blk < a.nblk_stride)
        a.block_scores[(int64_t)b * a.nblk_stride + blk] = bv;
    }
  } else {
    const int64_t slot = (int64_t)t * SWEEP_TILE + r;
    const int32_t blk = __ldg(a.pool + (int64_t)b * a.pool_nb + slot / BLOCK);
    const int64_t pos = (int64_t)blk * BLOCK + (r & (BLOCK - 1));
    const bool valid = blk >= 0 && pos < nv;
    srow[slot] = valid ? sc : -INFINITY;
  }
}

}  // namespace csa2
