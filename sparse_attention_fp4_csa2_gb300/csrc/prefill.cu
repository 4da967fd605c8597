// Chunked-prefill indexer: the lightning-indexer scores of many query tokens
// against the causally visible compressed entries of their sequence, on the
// 5th-generation tensor cores ("DeepSeek-V4.1-Flash - Architecture", sections
// 1-2: 20 encoder layers with CSA2 at m = 2; every chunk token indexes its own
// top-512 of the entries visible to it).
//
// Unlike decode, many queries share one key tile, so the contraction is a real
// GEMM and the kernel is bound by the tensor cores: per MMA, M = 128
// positions, N = 256 = 8 query tokens x 32 heads, K = 16; one 32 KB key tile
// feeds 8.4 MFLOP.  A work item is (a group of 8 consecutive tokens of one
// sequence, a range of key tiles); persistent CTAs take items round-robin.
// Warp 0 issues TMA loads (the group's 8 x 32 x 128 indexer queries once per
// item, key tiles into a 4-stage ring, the group's head weights into a double
// buffer), warp 1 issues the MMAs into two 256-column TMEM accumulators,
// warps 2-9 (two per TMEM lane quadrant, four tokens each) reduce each row to
// score(token, position) = sum_h w_h *
// ReLU(q_h . k) and write it, -inf where the position is not yet visible to
// the token (entry j is visible to the token at position g iff m*j + m-1 <= g).
#include "kernels.cuh"

namespace csa2 {

namespace {

constexpr int kStages = 4;
constexpr int kGroup = 8;                         // query tokens per MMA (N = 8 x 32 = 256)
constexpr int kN = kGroup * HI;                   // 256
constexpr int kTileBytes = SWEEP_TILE * DI * 2;   // 32 KB
constexpr int kQBytes = kN * DI * 2;              // 64 KB: two K-atoms of [256 rows][128 B]
constexpr int kWBytes = kN * 4;                   // 1 KB of head weights per group
constexpr int kEpiWarps = 8;                      // two warps per TMEM lane quadrant
constexpr int kThreads = 64 + kEpiWarps * 32;
constexpr uint32_t kIdesc = idesc_f16(/*bf16*/ 1, 0, 0, /*N*/ kN, /*M*/ SWEEP_TILE);

struct __align__(8) PrefillSmem {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t qfull, qempty;
  uint64_t wfull[2], wempty[2];
  uint64_t accfull[2], accempty[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
};

constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kTileBytes + kQBytes + 2 * kWBytes + sizeof(PrefillSmem);

__device__ __forceinline__ volatile uint32_t &abort_flag(PrefillSmem &S) {
  return *reinterpret_cast<volatile uint32_t *>(&S.abort);
}

struct Item {
  int64_t qg;    // first flattened query token of the group
  int32_t t0, t1;
};

__device__ __forceinline__ Item item_of(const PrefillIdxArgs &a, int64_t it) {
  const int64_t g = it / a.ranges;
  const int32_t r = (int32_t)(it % a.ranges);
  Item I;
  I.qg = a.q0 + g * kGroup;
  I.t0 = r * a.range_tiles;
  I.t1 = min(a.tiles, I.t0 + a.range_tiles);
  return I;
}

// entries visible to token i of its sequence
__device__ __forceinline__ int64_t visible(const PrefillIdxArgs &a, int64_t flat_q) {
  const int64_t g = a.first_pos + flat_q % a.tokens;
  int64_t n = (g + 1) / a.m;
  return n < a.cap ? n : a.cap;
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_indexer_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                           const PrefillIdxArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *kbuf = base;
  uint8_t *qbuf = base + (size_t)kStages * kTileBytes;
  float *wbuf = reinterpret_cast<float *>(qbuf + kQBytes);   // [2][256]
  PrefillSmem &S = *reinterpret_cast<PrefillSmem *>(qbuf + kQBytes + 2 * kWBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t n_items = a.groups * a.ranges;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], 1);
    }
    mbar_init(&S.qfull, 1);
    mbar_init(&S.qempty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.wfull[i], 1);
      mbar_init(&S.wempty[i], kEpiWarps * 32);
      mbar_init(&S.accfull[i], 1);
      mbar_init(&S.accempty[i], kEpiWarps * 32);
    }
    mbar_init(&S.mma_done, 1);
    abort_flag(S) = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_q);
  }
  // the inputs' producer is complete past here (programmatic launch)
  pdl_wait();
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, 2 * kN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      int64_t step = 0, j = 0;
      for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
        const Item I = item_of(a, it);
        const int64_t b = I.qg / a.tokens;
        if (!mbar_wait(&S.qempty, (uint32_t)((j & 1) ^ 1))) { abort_flag(S) = 1; break; }
        mbar_arrive_expect_tx(&S.qfull, kQBytes);
        tma_load_2d(qbuf, &tm_q, 0, (int32_t)(I.qg * HI), &S.qfull);
        tma_load_2d(qbuf + kQBytes / 2, &tm_q, 64, (int32_t)(I.qg * HI), &S.qfull);
        const int wb = (int)(j & 1);
        if (!mbar_wait(&S.wempty[wb], (uint32_t)(((j >> 1) & 1) ^ 1))) { abort_flag(S) = 1; break; }
        mbar_arrive_expect_tx(&S.wfull[wb], kWBytes);
        bulk_g2s(wbuf + wb * kN, a.w + I.qg * HI, kWBytes, &S.wfull[wb]);
        const int64_t nv_max = visible(a, I.qg + kGroup - 1);
        bool stop = false;
        for (int32_t t = I.t0; t < I.t1; ++t, ++step) {
          const int s = (int)(step % kStages);
          if (!mbar_wait(&S.empty[s], (uint32_t)(((step / kStages) & 1) ^ 1))) { stop = true; break; }
          uint8_t *dst = kbuf + (size_t)s * kTileBytes;
          if ((int64_t)t * SWEEP_TILE < nv_max) {
            const int32_t y = (int32_t)(b * a.cap + (int64_t)t * SWEEP_TILE);
            mbar_arrive_expect_tx(&S.full[s], kTileBytes);
            tma_load_2d(dst, &tm_k, 0, y, &S.full[s]);
            tma_load_2d(dst + kTileBytes / 2, &tm_k, 64, y, &S.full[s]);
          } else {
            mbar_arrive(&S.full[s]);
          }
        }
        if (stop) { abort_flag(S) = 1; break; }
      }
      // drain: the last phase of every stage and of the group buffers has landed
      for (int s = 0; s < kStages && s < step; ++s) {
        const int64_t last = s + ((step - 1 - s) / kStages) * kStages;
        mbar_wait(&S.full[s], (uint32_t)((last / kStages) & 1));
      }
      if (j > 0) mbar_wait(&S.qfull, (uint32_t)((j - 1) & 1));
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      int64_t step = 0, j = 0;
      const uint32_t kbase = smem_u32(kbuf), qa = smem_u32(qbuf);
      for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
        if (abort_flag(S)) break;
        const Item I = item_of(a, it);
        if (!mbar_wait(&S.qfull, (uint32_t)(j & 1))) { abort_flag(S) = 1; break; }
        bool stop = false;
        for (int32_t t = I.t0; t < I.t1; ++t, ++step) {
          const int s = (int)(step % kStages);
          const int acc = (int)(step & 1);
          if (!mbar_wait(&S.full[s], (uint32_t)((step / kStages) & 1)) ||
              !mbar_wait(&S.accempty[acc], (uint32_t)(((step >> 1) & 1) ^ 1))) { stop = true; break; }
          tc_fence_after();
          const uint32_t ka = kbase + (uint32_t)s * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < DI / 16; ++kk) {
            const uint64_t ad = smem_desc(ka + (kk >> 2) * (kTileBytes / 2) + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = smem_desc(qa + (kk >> 2) * (kQBytes / 2) + (kk & 3) * 32, 16, 1024);
            mma_f16(tmem + acc * kN, ad, bd, kIdesc, kk > 0 ? 1u : 0u);
          }
          mma_commit(&S.empty[s]);
          mma_commit(&S.accfull[acc]);
        }
        mma_commit(&S.qempty);
        if (stop) { abort_flag(S) = 1; break; }
      }
      pdl_release();   // the last item's MMAs are issued: the next kernel's CTAs may be dispatched
      mma_commit(&S.mma_done);
      mbar_wait(&S.mma_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warps 2..9: lane quadrant (warp & 3) of the tile, tokens 4*half .. 4*half+3
    const int quad = warp & 3, half = (warp - 2) >> 2;
    const int r = quad * 32 + lane;
    int64_t step = 0, j = 0;
    for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x, ++j) {
      const Item I = item_of(a, it);
      const int wb = (int)(j & 1);
      if (!mbar_wait(&S.wfull[wb], (uint32_t)((j >> 1) & 1))) { abort_flag(S) = 1; break; }
      // the head weights of two of this thread's four tokens stay in registers
      // for the whole item, halving the epilogue's shared-memory reads
      // (shared-memory bandwidth is what the MMAs run short of); the other
      // two are read per tile (the warps' register budget holds no more)
      const float *wv = wbuf + wb * kN;
      float wr[2][HI];
      {
        const float4 *w4 = reinterpret_cast<const float4 *>(wv + 4 * half * HI);
#pragma unroll
        for (int i = 0; i < HI / 2; ++i) {
          const float4 ww = w4[i];
          wr[i >> 3][(4 * i) & (HI - 1)] = ww.x;
          wr[i >> 3][((4 * i) & (HI - 1)) + 1] = ww.y;
          wr[i >> 3][((4 * i) & (HI - 1)) + 2] = ww.z;
          wr[i >> 3][((4 * i) & (HI - 1)) + 3] = ww.w;
        }
      }
      int32_t nv[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) nv[q] = (int32_t)visible(a, I.qg + 4 * half + q);
      float *srow = a.scores + (I.qg - a.q0 + 4 * half) * a.row_len;
      bool stop = false;
      for (int32_t t = I.t0; t < I.t1; ++t, ++step) {
        const int acc = (int)(step & 1);
        if (!mbar_wait(&S.accfull[acc], (uint32_t)((step >> 1) & 1))) { stop = true; break; }
        tc_fence_after();
        const int64_t pos = (int64_t)t * SWEEP_TILE + r;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int qq = 4 * half + q;
          uint32_t v[32];
          tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * kN + qq * HI), v);
          tmem_ld_wait();
          // four independent partial sums of w_h * ReLU(q_h . k), two per
          // packed fp32 FMA (heads h, h + 1 of every four in one, h + 2, h + 3
          // in the other; each lane as fmaf)
          const float4 *w4 = reinterpret_cast<const float4 *>(wv + qq * HI);
          uint64_t s01 = 0ull, s23 = 0ull;
#pragma unroll
          for (int h4 = 0; h4 < HI / 4; ++h4) {
            const float4 ww = q < 2 ? make_float4(wr[q & 1][4 * h4], wr[q & 1][4 * h4 + 1], wr[q & 1][4 * h4 + 2],
                                                  wr[q & 1][4 * h4 + 3])
                                    : w4[h4];
            s01 = f32x2_fma(f32x2_pack(ww.x, ww.y),
                            f32x2_pack(fmaxf(__uint_as_float(v[4 * h4 + 0]), 0.0f),
                                       fmaxf(__uint_as_float(v[4 * h4 + 1]), 0.0f)),
                            s01);
            s23 = f32x2_fma(f32x2_pack(ww.z, ww.w),
                            f32x2_pack(fmaxf(__uint_as_float(v[4 * h4 + 2]), 0.0f),
                                       fmaxf(__uint_as_float(v[4 * h4 + 3]), 0.0f)),
                            s23);
          }
          float s0, s1, s2, s3;
          f32x2_unpack(s01, s0, s1);
          f32x2_unpack(s23, s2, s3);
          const float sc = (s0 + s1) + (s2 + s3);
          srow[(int64_t)q * a.row_len + pos] = pos < nv[q] ? sc : -INFINITY;
        }
        tc_fence_before();
        mbar_arrive(&S.accempty[acc]);
      }
      mbar_arrive(&S.wempty[wb]);
      if (stop) { abort_flag(S) = 1; break; }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 2 * kN);
  }
}

}  // namespace

cudaError_t launch_prefill_indexer(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const PrefillIdxArgs &a,
                                   int num_sms, cudaStream_t stream, int *launches) {
  const int64_t n_items = a.groups * a.ranges;
  if (n_items <= 0) return cudaSuccess;
  cudaError_t err =
      cudaFuncSetAttribute(prefill_indexer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  const int grid = (int)(n_items < num_sms ? n_items : num_sms);
  const ProfileEvents &pe = profile_events(CSA2_KERNEL_PREFILL_INDEXER);
  if (pe.start && (err = record_profile_event(pe.start, stream)) != cudaSuccess) return err;
  err = launch_pdl(prefill_indexer_kernel, dim3(grid), dim3(kThreads), kSmemBytes, stream, 0u, tm_k, tm_q, a);
  if (err != cudaSuccess) return err;
  ++*launches;
  if (pe.stop) err = record_profile_event(pe.stop, stream);
  return err;
}

}  // namespace csa2
