// Exact top-K of each score row with one CTA per row (three per SM), for
// calls with many rows of up to 131,072 scores -- the index_topk = 512
// selection of every chunk token in prefill ("DeepSeek-V4.1-Flash -
// Architecture", sections 2 and 3) -- where throughput over the rows, not
// the latency of one row, sets the time.  Same contract as
// the cluster kernel: scores become order-preserving 32-bit keys (-inf and
// NaN mark an invalid slot and are never taken), the k largest keys win,
// keys equal on all 32 bits go to the lower index, the selection is written
// in index order (mapped through the HSI pool for Reindex rows) and padded
// with -1.
//
// No cluster barriers, no global scratch:
//   1. sample: the first 512 scores of every 4096 (an eighth of the row,
//      plain coalesced loads); two histogram levels (key bits 31..21, then
//      20..10 inside the threshold bin) give a low threshold t_low with about
//      twice the sample's share of k above it;
//   2. filter: the row streams through two 16 KB shared-memory stages
//      filled by bulk copies one stage ahead; every key >= t_low goes to the
//      candidate list in index order (per-warp ballots and one scan of the
//      warp counts per stage give every key its slot: no per-key atomics);
//   3. when the list did not overflow and holds every key of the top k (at
//      least k keys, or every valid key), three radix levels (11, 11 and 10
//      key bits) over the list find the k-th largest key T and how many keys
//      equal to T are still needed; one ordered pass writes the keys above T
//      and the first such ties;
//   4. otherwise the same levels and the ordered pass run over the whole row
//      (streamed through the ring each time): exact for any input, only
//      slower.
#include "kernels.cuh"

namespace csa2 {

namespace {

constexpr int kRT = 512;                 // threads per CTA
constexpr int kRW = kRT / 32;
constexpr int kChunk = 4096;             // scores per ring stage (16 KB)
constexpr int kStages = 2;
constexpr int kRCand = 4096;             // candidate list
constexpr int kRBins = 2048;
constexpr int kSampleLen = 512;          // sampled scores at the head of every chunk (1/8)
constexpr int kRowMax = 131072;

struct __align__(128) RowTopkSmem {
  float ring[kStages][kChunk];
  uint32_t ckey[kRCand];
  int32_t cidx[kRCand];
  uint32_t hist[kRBins];
  uint64_t full[kStages];
  uint32_t seg[2 * kRW];       // per (half, warp) counts of a stage, then their exclusive prefix
  uint32_t seg_total;
  uint32_t bscan[kRW];
  int thr;
  uint32_t above, total;
};

constexpr size_t kRowSmem = sizeof(RowTopkSmem) + 128;
static_assert(3 * (kRowSmem + 1024) <= 233472, "three CTAs must fit on an SM");

__device__ __forceinline__ uint32_t row_key(float v) {
  return (v == -INFINITY || v != v) ? 0u : f32_key(v);
}

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Histogram add aggregated over the warp's equal bins (kRBins: none); every
// lane of the warp calls it.
__device__ __forceinline__ void hist_agg(uint32_t *h, uint32_t bin) {
  const uint32_t peers = __match_any_sync(0xffffffffu, bin);
  if (bin < kRBins && (threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&h[bin], (uint32_t)__popc(peers));
}

// Within-warp exclusive ranks of four flags per lane in (lane, e) order, and
// the warp's count.
__device__ __forceinline__ uint32_t warp_ranks(const bool (&f)[4], uint32_t (&rank)[4]) {
  const uint32_t lt = lanemask_lt();
  uint32_t m[4], before = 0, tot = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    m[e] = __ballot_sync(0xffffffffu, f[e]);
    before += __popc(m[e] & lt);
    tot += __popc(m[e]);
  }
  uint32_t own = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    rank[e] = before + own;
    own += f[e] ? 1u : 0u;
  }
  return tot;
}

// Exclusive prefix of the (half, warp) segment counts in (half, warp) order
// -- the index order of a stage -- and their total.  Two CTA barriers.
__device__ __forceinline__ void seg_scan(RowTopkSmem &S, uint32_t c0, uint32_t c1, uint32_t &b0, uint32_t &b1,
                                         uint32_t &total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0) {
    S.seg[w] = c0;
    S.seg[kRW + w] = c1;
  }
  __syncthreads();
  if (w == 0) {
    const uint32_t v = S.seg[lane];
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    S.seg[lane] = incl - v;
    if (lane == 31) S.seg_total = incl;
  }
  __syncthreads();
  b0 = S.seg[w];
  b1 = S.seg[kRW + w];
  total = S.seg_total;
}

// Threshold bin of hist[0 .. bins) for `need` keys counted from the top:
// thr = -1 when all of them fit (total <= need); above = keys in higher bins.
// Clears hist.  Ends with the CTA synchronised.
__device__ void row_threshold(RowTopkSmem &S, uint32_t need, int bins) {
  constexpr int kPer = kRBins / kRT;   // 4 bins per thread
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  uint32_t c[kPer], loc = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    const int b = bins - 1 - (kPer * tid + j);
    c[j] = b >= 0 ? S.hist[b] : 0u;
    loc += c[j];
  }
  uint32_t incl = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) S.bscan[w] = incl;
  __syncthreads();
  uint32_t wbase = 0, total = 0;
#pragma unroll
  for (int i = 0; i < kRW; ++i) {
    const uint32_t x = S.bscan[i];
    wbase += i < w ? x : 0u;
    total += x;
  }
  uint32_t before = wbase + incl - loc;
  if (tid == 0) {
    S.thr = -1;
    S.above = total;
    S.total = total;
  }
  __syncthreads();
  if (total > need) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = bins - 1 - (kPer * tid + j);
      if (b >= 0 && before < need && before + c[j] >= need) {
        S.thr = b;
        S.above = before;
      }
      before += c[j];
    }
  }
#pragma unroll
  for (int j = 0; j < kPer; ++j) S.hist[kPer * tid + j] = 0;
  __syncthreads();
}

// Level-L predicate and digit of the radix select: level 0 every valid key,
// bits 31..21; level 1 keys whose bits 31..21 equal the prefix, bits 20..10;
// level 2 keys whose bits 31..10 equal the prefix, bits 9..0.
__device__ __forceinline__ uint32_t level_bin(uint32_t key, int level, uint32_t prefix) {
  if (!key) return kRBins;
  if (level == 0) return key >> 21;
  if (level == 1) return (key >> 21) == prefix ? ((key >> 10) & 2047u) : (uint32_t)kRBins;
  return (key >> 10) == prefix ? (key & 1023u) : (uint32_t)kRBins;
}

// Streams chunks [0, nch) of the row through the ring: f(keys, base) per
// chunk, keys[h][e] the key at base + 2048 h + 4 tid + e (0 past n).  `g` is
// the running count of chunks through the ring (the stage and barrier phase
// of every chunk); thread 0 refills a stage after the CTA barrier that ends
// its chunk.
template <typename F>
__device__ __forceinline__ void stream_row(RowTopkSmem &S, const float *vals, int64_t n, uint32_t &g, F &&f) {
  const int tid = threadIdx.x;
  const int nch = (int)((n + kChunk - 1) / kChunk);
  auto issue = [&](int c, uint32_t gi) {
    const int s = (int)(gi % kStages);
    const uint32_t bytes = (uint32_t)(4 * min((int64_t)kChunk, n - (int64_t)c * kChunk));
    mbar_arrive_expect_tx(&S.full[s], bytes);
    bulk_g2s(S.ring[s], vals + (int64_t)c * kChunk, bytes, &S.full[s]);
  };
  if (tid == 0)
    for (int c = 0; c < nch && c < kStages; ++c) issue(c, g + (uint32_t)c);
#pragma unroll 1
  for (int c = 0; c < nch; ++c, ++g) {
    const int s = (int)(g % kStages);
    (void)mbar_wait(&S.full[s], (g / kStages) & 1u);
    const int64_t base = (int64_t)c * kChunk;
    uint32_t keys[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int o = 2048 * h + 4 * tid;
      const float4 v = *reinterpret_cast<const float4 *>(&S.ring[s][o]);
      const bool in = base + o < n;   // n % 4 == 0: a float4 is wholly in or out
      keys[h][0] = in ? row_key(v.x) : 0u;
      keys[h][1] = in ? row_key(v.y) : 0u;
      keys[h][2] = in ? row_key(v.z) : 0u;
      keys[h][3] = in ? row_key(v.w) : 0u;
    }
    f(keys, base);
    __syncthreads();   // every thread is done with the stage
    if (tid == 0 && c + kStages < nch) issue(c + kStages, g + kStages);
  }
}

// The candidate list read in the same stage layout (chunks of 4096 entries).
template <typename F>
__device__ __forceinline__ void stream_cands(RowTopkSmem &S, uint32_t cnt, F &&f) {
  const int tid = threadIdx.x;
#pragma unroll 1
  for (uint32_t base = 0; base < cnt; base += kChunk) {
    uint32_t keys[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t o = base + 2048 * h + 4 * tid;
      const uint4 k4 = o < cnt ? *reinterpret_cast<const uint4 *>(&S.ckey[o]) : make_uint4(0, 0, 0, 0);
      // entries past cnt inside the last float4 hold stale keys: mask them
      keys[h][0] = o + 0 < cnt ? k4.x : 0u;
      keys[h][1] = o + 1 < cnt ? k4.y : 0u;
      keys[h][2] = o + 2 < cnt ? k4.z : 0u;
      keys[h][3] = o + 3 < cnt ? k4.w : 0u;
    }
    f(keys, (int64_t)base);
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kRT, 1) topk_row_kernel(const TopkRows r) {
  extern __shared__ uint8_t smem_raw[];
  RowTopkSmem &S =
      *reinterpret_cast<RowTopkSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int tid = threadIdx.x;
  const int row = blockIdx.x;
  const float *vals = r.vals + (int64_t)row * r.row_stride;
  const int64_t n = r.row_len;
  const uint32_t k = (uint32_t)r.k;

  // the whole row heads for L2 at once (the filter reads it again after the
  // sample levels): one bulk prefetch per chunk
  if (tid == 0)
    for (int64_t c = 0; c * kChunk < n; ++c)
      prefetch_l2_bulk(vals + c * kChunk, (uint32_t)(4 * min((int64_t)kChunk, n - c * kChunk)));
  if (tid < kStages) mbar_init(&S.full[tid], 1);
  for (int i = tid; i < kRBins; i += kRT) S.hist[i] = 0;
  fence_barrier_init();
  __syncthreads();

  // ------------------------------------------------------------ 1. sample
  // The first kSampleLen scores of every chunk; eight float4 per thread in
  // flight per batch.
  const int64_t nch = (n + kChunk - 1) / kChunk;
  const int64_t ns4 = nch * (kSampleLen / 4);
  auto sample = [&](int level, uint32_t b0) {
#pragma unroll 1
    for (int64_t q0 = 0; q0 < ns4; q0 += 8 * kRT) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t q = q0 + tid + (int64_t)j * kRT;
        const int64_t p = (q / (kSampleLen / 4)) * kChunk + 4 * (q % (kSampleLen / 4));
        v[j] = (q < ns4 && p < n) ? __ldcg(reinterpret_cast<const float4 *>(vals + p))
                                  : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float x[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t key = row_key(x[e]);
          if (level == 0) {
            hist_agg(S.hist, key ? key >> 21 : (uint32_t)kRBins);
          } else if (key && (key >> 21) == b0) {
            atomicAdd(&S.hist[(key >> 10) & 2047u], 1u);
          }
        }
      }
    }
    __syncthreads();
  };
  const uint32_t need_s = k / 4 + 16;   // about twice the sample's share of k
  uint32_t t_low = 1;                   // 1: every valid key
  sample(0, 0);
  row_threshold(S, need_s, kRBins);
  if (S.thr >= 0) {
    const uint32_t b0 = (uint32_t)S.thr, above0 = S.above;
    sample(1, b0);
    row_threshold(S, need_s - above0, kRBins);
    t_low = S.thr < 0 ? (b0 << 21) : ((b0 << 21) | ((uint32_t)S.thr << 10));
  }

  // ------------------------------------------------------------ 2. filter
  uint32_t g = 0;        // chunks through the ring so far
  uint32_t ccount = 0;   // candidates (may exceed the list: overflow)
  stream_row(S, vals, n, g, [&](uint32_t(&keys)[2][4], int64_t base) {
    uint32_t rk[2][4], cnt[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      bool f[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) f[e] = keys[h][e] >= t_low;
      cnt[h] = warp_ranks(f, rk[h]);
    }
    uint32_t b0, b1, tot;
    seg_scan(S, cnt[0], cnt[1], b0, b1, tot);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (keys[h][e] >= t_low) {
          const uint32_t pos = ccount + (h ? b1 : b0) + rk[h][e];
          if (pos < kRCand) {
            S.ckey[pos] = keys[h][e];
            S.cidx[pos] = (int32_t)(base + 2048 * h + 4 * tid + e);
          }
        }
    ccount += tot;
  });
  // the list holds every key of the top k when it did not overflow and has
  // at least k keys, or every valid key of the row (t_low = 1)
  const bool from_list = ccount <= (uint32_t)kRCand && (ccount >= k || t_low == 1);

  // --------------------------------------------------------- 3./4. select
  // T: the k-th largest key; keys above T are taken, and of the keys equal
  // to T the first tie_need in index order.  T = 0 takes every valid key.
  uint32_t T = 0, tie_need = 0;
  {
    uint32_t need = k, prefix = 0;
#pragma unroll 1
    for (int L = 0; L < 3; ++L) {
      auto hist = [&](uint32_t(&keys)[2][4], int64_t) {
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const uint32_t bin = level_bin(keys[h][e], L, prefix);
            if (L == 0)
              hist_agg(S.hist, bin);
            else if (bin < kRBins)
              atomicAdd(&S.hist[bin], 1u);
          }
      };
      if (from_list)
        stream_cands(S, ccount, hist);
      else
        stream_row(S, vals, n, g, hist);
      row_threshold(S, need, L == 2 ? 1024 : kRBins);
      const int thr = S.thr;
      const uint32_t above = S.above;
      const int shift = L == 0 ? 21 : L == 1 ? 10 : 0;
      if (thr < 0) {
        // everything matching fits: at level 0 every valid key; deeper, the
        // previous bin holds exactly the count still needed
        T = L == 0 ? 0u : (prefix << (shift + (L == 1 ? 11 : 10)));
        tie_need = L == 0 ? 0u : need;
        break;
      }
      need -= above;
      prefix = L == 0 ? (uint32_t)thr : (prefix << (L == 1 ? 11 : 10)) | (uint32_t)thr;
      if (L == 2) {
        T = prefix;
        tie_need = need;
      }
    }
  }

  int32_t *out = r.out + (int64_t)row * r.k;
  const int32_t *pool = r.pool ? r.pool + (int64_t)row * r.pool_stride : nullptr;
  uint32_t sel_before = 0, tie_before = 0;
  auto emit = [&](uint32_t(&keys)[2][4], int64_t base) {
    bool te[2][4], any_tie = false;
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        te[h][e] = keys[h][e] == T && keys[h][e] != 0u;
        any_tie |= te[h][e];
      }
    uint32_t trk[2][4] = {}, tb0 = 0, tb1 = 0, ttot = 0;
    if (__syncthreads_or(any_tie)) {
      uint32_t tc[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) tc[h] = warp_ranks(te[h], trk[h]);
      seg_scan(S, tc[0], tc[1], tb0, tb1, ttot);
    }
    bool fl[2][4];
    uint32_t srk[2][4], sc[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        fl[h][e] = keys[h][e] > T || (te[h][e] && tie_before + (h ? tb1 : tb0) + trk[h][e] < tie_need);
      sc[h] = warp_ranks(fl[h], srk[h]);
    }
    uint32_t sb0, sb1, stot;
    seg_scan(S, sc[0], sc[1], sb0, sb1, stot);
#pragma unroll
    for (int h = 0; h < 2; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (fl[h][e]) {
          const uint32_t pos = sel_before + (h ? sb1 : sb0) + srk[h][e];
          const int64_t o = base + 2048 * h + 4 * tid + e;
          const int32_t v = from_list ? S.cidx[o] : (int32_t)o;
          if (pos < k) out[pos] = pool ? __ldg(pool + v / BLOCK) * BLOCK + (v & (BLOCK - 1)) : v;
        }
    sel_before += stot;
    tie_before += ttot;
  };
  if (from_list)
    stream_cands(S, ccount, emit);
  else
    stream_row(S, vals, n, g, emit);
  for (uint32_t i = min(sel_before, k) + tid; i < k; i += kRT) out[i] = -1;
}

}  // namespace

bool topk_row_supported(const TopkRows &r) {
  return r.k >= 1 && r.k <= 2048 && r.row_len >= 0 && r.row_len <= kRowMax && r.row_len % 4 == 0 &&
         r.row_stride % 4 == 0 && (reinterpret_cast<uintptr_t>(r.vals) & 15u) == 0;
}

cudaError_t launch_topk_row(const TopkRows &r, cudaStream_t stream, int *launches, bool profiled) {
  if (r.rows <= 0) return cudaSuccess;
  if (!topk_row_supported(r)) return cudaErrorInvalidValue;
  cudaError_t err = cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRowSmem);
  if (err != cudaSuccess) return err;
  static const ProfileEvents kNone;
  const ProfileEvents &pe = profiled ? profile_events(CSA2_KERNEL_TOPK) : kNone;
  if (pe.start && (err = record_profile_event(pe.start, stream)) != cudaSuccess) return err;
  topk_row_kernel<<<(unsigned)r.rows, kRT, kRowSmem, stream>>>(r);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  ++*launches;
  if (pe.stop) err = record_profile_event(pe.stop, stream);
  return err;
}


namespace {
int g_topk_choice = 0;
}  // namespace

void set_topk_choice(int which) { g_topk_choice = which; }

cudaError_t launch_topk(const TopkRows &r, cudaStream_t stream, int *launches, bool profiled) {
  if (g_topk_choice == 2) return launch_topk_row(r, stream, launches, profiled);   // strict: no fallback
  // automatic: one CTA per row once the rows fill every SM twice (the cluster
  // kernel then runs a single CTA per row too, with a longer chain per row);
  // fewer rows go to a cluster per row, which spreads each row over SMs
  if (g_topk_choice == 0 && topk_row_supported(r)) {
    static int sms = 0;
    if (!sms) {
      int dev = 0;
      if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) !=
                                                    cudaSuccess)
        sms = 1 << 20;
    }
    if (r.rows >= 2 * sms) return launch_topk_row(r, stream, launches, profiled);
  }
  return launch_topk_cluster(r, stream, launches, profiled);
}

}  // namespace csa2
