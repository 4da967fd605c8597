// Lightning-indexer sweep on the 5th-generation tensor cores.
//
// score(n) = sum_h w_h * ReLU(q_h . k_n), 32 heads x 128 dims ("DeepSeek-V4.1-
// Flash - Architecture", section 2, main attention settings), over
//   Full:    every position of the sequence up to n_vis (linear in context,
//            "the first Full layer still scans the full range", section 3);
//   Reindex: the positions of the HSI candidate pool only (2048 blocks x 8,
//            "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache
//            Compression", section 2.3.4).
// The Full sweep also writes the HSI block scores (max -- or sum -- of each
// block of 8 visible scores; -inf past n_vis).
//
// Per 128-position tile: S[128 x 32] = K_tile[128 x 128] . Q^T (tcgen05.mma
// kind::f16, bf16 operands from 128B-swizzled shared memory, fp32 accumulator
// in TMEM), then an epilogue reduces the 32 head columns of each row.  The
// sweep reads 256 B per position and does 8192 flops on it (32 flop/B), so it
// is bound by HBM; the tensor cores only keep it from becoming bound by the
// CUDA-core FMA rate.
//
// Persistent, warp-specialised CTA (one per SM): warp 0 issues TMA loads of
// the K tiles into a ring of shared-memory stages, warp 1 issues the MMAs into
// two TMEM accumulators, warps 2-5 drain the accumulators (and, when the
// cluster top-K follows, count every score's key in the row's histogram; see
// HistSegments).  Every CTA owns a contiguous run of (sequence, tile) work
// items.
#include "pipeline.cuh"

namespace csa2 {

namespace {

constexpr int kStages = 6;
constexpr int kTileBytes = SWEEP_TILE * DI * 2;  // 32 KB: two 16 KB K-atoms of [128 rows][128 B]
constexpr int kQBytes = HI * DI * 2;             // 8 KB: two 4 KB K-atoms of [32 rows][128 B]
constexpr int kThreads = 192;
constexpr uint32_t kIdesc = idesc_f16(/*bf16*/ 1, /*A K-major*/ 0, /*B K-major*/ 0, /*N*/ HI, /*M*/ SWEEP_TILE);

struct __align__(8) SweepSmem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t qfull[2];
  uint64_t qempty[2];
  uint64_t accfull[2];
  uint64_t accempty[2];
  uint64_t mma_done;
  uint64_t hseg[2];    // histogram slot: the four epilogue warps are done adding to it
  uint64_t hfree[2];   // histogram slot: flushed and cleared
  uint32_t tmem_base;
  uint32_t abort;
};

__device__ __forceinline__ volatile uint32_t &abort_flag(SweepSmem &S) {
  return *reinterpret_cast<volatile uint32_t *>(&S.abort);
}

constexpr size_t kHistOff = (sizeof(SweepSmem) + 15) / 16 * 16;   // after the control block
constexpr size_t kSmemBytes =
    1024 /*align slack*/ + (size_t)kStages * kTileBytes + 2 * kQBytes + kHistOff + 2 * kHistWords * 4;
constexpr int kSegTiles = 256;   // 128 keys a tile: a segment's counts stay below 2^16
static_assert(kSmemBytes <= 232448, "shared memory of one CTA");

__device__ __forceinline__ int32_t clamp_nvis(const int32_t *n_vis, int b, int64_t n_max) {
  int32_t v = __ldg(n_vis + b);
  if (v < 0 || v > n_max) {
    set_error(CSA2_DEV_ERR_NVIS);
    v = v < 0 ? 0 : (int32_t)n_max;
  }
  return v;
}

// Row r of tile t of sequence b: score = sum_h w_h ReLU(dot_h) ("DeepSeek-
// V4.1-Flash - Architecture", section 2), -inf where the position is not
// visible; the Full sweep also writes the max (or sum) over each block of 8
// ("DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression", 2.3.4),
// and counts the score's key in the row's histogram when one is kept.
// Called by all 32 lanes of a warp (the block reduction shuffles).
template <bool kPool>
__device__ __forceinline__ void sweep_store_row(const SweepArgs &a, int b, int t, int r, int lane, int32_t nv,
                                                const float (&wv)[HI], const uint32_t (&v)[32], uint32_t *hs) {
  float sc = 0.0f;
#pragma unroll
  for (int h = 0; h < HI; ++h) sc = fmaf(wv[h], fmaxf(__uint_as_float(v[h]), 0.0f), sc);
  float *srow = a.scores + (int64_t)b * a.row_len;
  float stored;
  if (!kPool) {
    const int64_t pos = (int64_t)t * SWEEP_TILE + r;
    const bool valid = pos < nv;
    stored = valid ? sc : -INFINITY;
    srow[pos] = stored;
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
    stored = valid ? sc : -INFINITY;
    srow[slot] = stored;
  }
  if (hs) hist_count(hs, stored);
}

template <bool kPool>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_sweep_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                         const SweepArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *kbuf = base;                                  // kStages x 32 KB, 1024-aligned
  uint8_t *qbuf = base + (size_t)kStages * kTileBytes;   // 2 x 8 KB
  SweepSmem &S = *reinterpret_cast<SweepSmem *>(qbuf + 2 * kQBytes);
  // the rows' histogram slots (two, by segment parity) when the top-K takes one
  uint32_t *hist_s = reinterpret_cast<uint32_t *>(qbuf + 2 * kQBytes + kHistOff);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t total = (int64_t)a.batch * a.tiles_per_seq;
  const int64_t it0 = total * blockIdx.x / gridDim.x;
  const int64_t it1 = total * (blockIdx.x + 1) / gridDim.x;
  const int n_tiles = (int)(it1 - it0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.qfull[i], 1);
      mbar_init(&S.qempty[i], 1);
      mbar_init(&S.accfull[i], 1);
      mbar_init(&S.accempty[i], 4 * 32);
    }
    mbar_init(&S.mma_done, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.hseg[i], 4);   // the four epilogue warps
      mbar_init(&S.hfree[i], 4);
    }
    abort_flag(S) = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_q);
  }
  if (a.hist)
    for (int i = threadIdx.x; i < 2 * kHistWords; i += kThreads) hist_s[i] = 0u;   // both slots
  // the inputs' producer is complete past here (programmatic launch)
  pdl_wait();
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 64);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Full tiles: lane 0 alone; pool tiles (Reindex): the whole warp, a lane
    // per pool block
    if (!kPool) {
      if (lane == 0) {
        // K rows are read once: evict them first, so that the scores this
        // kernel writes stay in L2 for the top-K that reads them next
        const uint64_t pol = l2_policy_evict_first();
        int prev_b = -1, qi = -1;
        int32_t nv = 0;
        int64_t n_issued = 0;
        for (int64_t it = it0; it < it1; ++it) {
          const int b = (int)(it / a.tiles_per_seq);
          const int t = (int)(it % a.tiles_per_seq);
          if (b != prev_b) {
            if (qi >= 0 && abort_flag(S)) break;
            ++qi;
            const int qs = qi & 1;
            if (!mbar_wait(&S.qempty[qs], ((qi >> 1) & 1) ^ 1)) { abort_flag(S) = 1; break; }
            mbar_arrive_expect_tx(&S.qfull[qs], kQBytes);
            tma_load_2d(qbuf + qs * kQBytes, &tm_q, 0, b * HI, &S.qfull[qs]);
            tma_load_2d(qbuf + qs * kQBytes + kQBytes / 2, &tm_q, 64, b * HI, &S.qfull[qs]);
            nv = clamp_nvis(a.n_vis, b, a.n_max);
            prev_b = b;
          }
          const int64_t li = it - it0;
          const int s = (int)(li % kStages);
          const uint32_t ph = (uint32_t)((li / kStages) & 1);
          if (!mbar_wait(&S.empty[s], ph ^ 1)) { abort_flag(S) = 1; break; }
          uint8_t *dst = kbuf + (size_t)s * kTileBytes;
          const int64_t row0 = (int64_t)b * a.cap;
          if ((int64_t)t * SWEEP_TILE < nv) {
            mbar_arrive_expect_tx(&S.full[s], kTileBytes);
            tma_load_2d_hint(dst, &tm_k, 0, (int32_t)(row0 + (int64_t)t * SWEEP_TILE), &S.full[s], pol);
            tma_load_2d_hint(dst + kTileBytes / 2, &tm_k, 64, (int32_t)(row0 + (int64_t)t * SWEEP_TILE), &S.full[s],
                             pol);
          } else {
            mbar_arrive(&S.full[s]);
          }
          ++n_issued;
        }
        // Drain: every load this thread issued has landed before the CTA can
        // exit (returns at once unless a wait above gave up).
        for (int s = 0; s < kStages && s < n_issued; ++s) {
          const int64_t last = s + ((n_issued - 1 - s) / kStages) * kStages;
          mbar_wait(&S.full[s], (uint32_t)((last / kStages) & 1));
        }
        if (qi >= 0) mbar_wait(&S.qfull[qi & 1], (qi >> 1) & 1);
      }
    } else {
      // lane 0 drives the rings; lane j fetches pool block j and its 8 rows
      const uint64_t pol = l2_policy_evict_first();
      int prev_b = -1, q_issued = 0;
      int32_t nv = 0;
      int n_issued = 0;
      TileCursor cur(it0, a.tiles_per_seq);
      Ring<kStages> kr;
      for (int li = 0; li < n_tiles; ++li, cur.next(), kr.next()) {
        const int b = cur.b, t = cur.t;
        int ok = 1;
        if (b != prev_b) {
          if (lane == 0) {
            const int qs = q_issued & 1;
            if (q_issued > 0 && abort_flag(S)) {
              ok = 0;
            } else if (!mbar_wait(&S.qempty[qs], ((q_issued >> 1) & 1) ^ 1)) {
              abort_flag(S) = 1;
              ok = 0;
            } else {
              mbar_arrive_expect_tx(&S.qfull[qs], kQBytes);
              tma_load_2d(qbuf + qs * kQBytes, &tm_q, 0, b * HI, &S.qfull[qs]);
              tma_load_2d(qbuf + qs * kQBytes + kQBytes / 2, &tm_q, 64, b * HI, &S.qfull[qs]);
              nv = clamp_nvis(a.n_vis, b, a.n_max);
            }
          }
          if (!warp_bcast<kPool>(ok)) break;
          nv = warp_bcast<kPool>(nv);
          ++q_issued;
          prev_b = b;
        }
        const int s = kr.slot;
        if (lane == 0 && !mbar_wait(&S.empty[s], kr.phase ^ 1)) {
          abort_flag(S) = 1;
          ok = 0;
        }
        if (!warp_bcast<kPool>(ok)) break;
        uint8_t *dst = kbuf + (size_t)s * kTileBytes;
        const int64_t row0 = (int64_t)b * a.cap;
        constexpr int kBlocks = SWEEP_TILE / BLOCK;   // pool blocks per tile
        const int64_t nblk_vis = ((int64_t)nv + BLOCK - 1) / BLOCK;
        const int32_t blk =
            lane < kBlocks ? __ldg(a.pool + (int64_t)b * a.pool_nb + (int64_t)t * kBlocks + lane) : -1;
        const bool v = blk >= 0 && blk < nblk_vis;
        if (lane < kBlocks && !v && blk >= nblk_vis && (int64_t)blk * BLOCK >= a.n_max) set_error(CSA2_DEV_ERR_POOL);
        const uint32_t valid = __ballot_sync(0xffffffffu, v);
        if (valid) {
          if (lane == 0) mbar_arrive_expect_tx(&S.full[s], (uint32_t)__popc(valid) * (BLOCK * DI * 2));
          __syncwarp();
          if (v) {
            const int32_t y = (int32_t)(row0 + (int64_t)blk * BLOCK);
            tma_load_2d_hint(dst + lane * 1024, &tm_k, 0, y, &S.full[s], pol);
            tma_load_2d_hint(dst + kTileBytes / 2 + lane * 1024, &tm_k, 64, y, &S.full[s], pol);
          }
        } else if (lane == 0) {
          mbar_arrive(&S.full[s]);
        }
        ++n_issued;
      }
      // Drain: every load this warp issued has landed before the CTA can exit
      // (returns at once unless a wait above gave up).
      if (lane == 0) {
        for (int s = 0; s < kStages && s < n_issued; ++s) {
          const int last = s + ((n_issued - 1 - s) / kStages) * kStages;
          mbar_wait(&S.full[s], (uint32_t)((last / kStages) & 1));
        }
        if (q_issued > 0) mbar_wait(&S.qfull[(q_issued - 1) & 1], ((q_issued - 1) >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int prev_b = -1, qi = -1;
      const uint32_t kbase = smem_u32(kbuf), qbase = smem_u32(qbuf);
      for (int64_t it = it0; it < it1; ++it) {
        if (abort_flag(S)) break;
        const int b = (int)(it / a.tiles_per_seq);
        if (b != prev_b) {
          if (qi >= 0) mma_commit(&S.qempty[qi & 1]);
          ++qi;
          if (!mbar_wait(&S.qfull[qi & 1], (qi >> 1) & 1)) { abort_flag(S) = 1; break; }
          prev_b = b;
        }
        const int64_t li = it - it0;
        const int s = (int)(li % kStages);
        const uint32_t ph = (uint32_t)((li / kStages) & 1);
        const int acc = (int)(li & 1);
        const uint32_t aph = (uint32_t)((li >> 1) & 1);
        if (!mbar_wait(&S.full[s], ph)) { abort_flag(S) = 1; break; }
        if (!mbar_wait(&S.accempty[acc], aph ^ 1)) { abort_flag(S) = 1; break; }
        tc_fence_after();
        const uint32_t ka = kbase + (uint32_t)s * kTileBytes;
        const uint32_t qa = qbase + (uint32_t)(qi & 1) * kQBytes;
#pragma unroll
        for (int kk = 0; kk < DI / 16; ++kk) {
          const uint64_t ad = smem_desc(ka + (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = smem_desc(qa + (kk >> 2) * (kQBytes / 2) + (kk & 3) * 32, 16, 1024);
          mma_f16(tmem + acc * HI, ad, bd, kIdesc, kk > 0 ? 1u : 0u);
        }
        mma_commit(&S.empty[s]);
        mma_commit(&S.accfull[acc]);
      }
      pdl_release();   // the last tile's MMAs are issued: the next kernel's CTAs may be dispatched
      // every MMA has completed before TMEM is released
      mma_commit(&S.mma_done);
      mbar_wait(&S.mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;               // TMEM lane quadrant this warp may read
    const int r = quad * 32 + lane;          // row of the tile = TMEM lane
    int prev_b = -1;
    int32_t nv = 0;
    float wv[HI];
    HistSegments hseg(S.hseg, S.hfree, hist_s, a.hist, kSegTiles, quad, lane);
    for (int64_t it = it0; it < it1; ++it) {
      if (abort_flag(S)) break;
      const int b = (int)(it / a.tiles_per_seq);
      const int t = (int)(it % a.tiles_per_seq);
      hseg.tile(b);
      if (b != prev_b) {
#pragma unroll
        for (int h = 0; h < HI; ++h) wv[h] = __ldg(a.w + (int64_t)b * HI + h);
        nv = clamp_nvis(a.n_vis, b, a.n_max);
        prev_b = b;
      }
      const int64_t li = it - it0;
      const int acc = (int)(li & 1);
      const uint32_t aph = (uint32_t)((li >> 1) & 1);
      if (!mbar_wait(&S.accfull[acc], aph)) { abort_flag(S) = 1; break; }
      tc_fence_after();
      uint32_t v[32];
      tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * HI), v);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&S.accempty[acc]);
      sweep_store_row<kPool>(a, b, t, r, lane, nv, wv, v, hseg.slot());
    }
    hseg.finish();
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

}  // namespace

cudaError_t launch_indexer_sweep(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const SweepArgs &a, int num_sms,
                                 cudaStream_t stream, int *launches) {
  const int64_t total = (int64_t)a.batch * a.tiles_per_seq;
  if (total <= 0) return cudaSuccess;
  const int grid = (int)(total < num_sms ? total : num_sms);
  const ProfileEvents &pe = profile_events(CSA2_KERNEL_INDEXER_SWEEP);
  cudaError_t err;
  if (pe.start && (err = record_profile_event(pe.start, stream)) != cudaSuccess) return err;
  if (a.pool) {
    err = cudaFuncSetAttribute(indexer_sweep_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    err = launch_pdl(indexer_sweep_kernel<true>, dim3(grid), dim3(kThreads), kSmemBytes, stream, 0u, tm_k, tm_q, a);
  } else {
    err = cudaFuncSetAttribute(indexer_sweep_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    err = launch_pdl(indexer_sweep_kernel<false>, dim3(grid), dim3(kThreads), kSmemBytes, stream, 0u, tm_k, tm_q, a);
  }
  if (err != cudaSuccess) return err;
  ++*launches;
  if (pe.stop) err = record_profile_event(pe.stop, stream);
  return err;
}

}  // namespace csa2
