// Exact top-K of each score row with one CTA per row (two per SM), for
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
//      plain coalesced loads); a histogram of key bits 31..21 gives a low
//      threshold t_low with about twice the sample's share of k above it --
//      refined by a second level (bits 20..10 inside the threshold bin) when
//      that bin would bring more candidates than the list should hold;
//   2. filter: the row read once with coalesced loads, eight float4 per
//      thread in flight; a float compare against the smallest score with a
//      key >= t_low keeps the candidates (32 flags per thread as one mask,
//      one warp scan of the counts), whose positions go to the warp's own
//      segment of a list (its count kept in a register: no atomics); the
//      segments are then packed, keys read again, into one 4,096-entry list
//      in no particular order;
//   3. when the list did not overflow and holds every key of the top k (at
//      least k keys, or every valid key), three radix levels (11, 11 and 10
//      key bits) over it find the k-th largest key T and how many keys equal
//      to T are still needed; the keys above T and the lowest-index ties
//      (ranked by comparing indices) are gathered and written in index
//      order through a bitmap of the row (one bit per position);
//   4. otherwise -- the list overflowed, missed part of the top k, or holds
//      more than 256 ties of T -- the levels (if needed) and an ordered pass
//      run over the whole row streamed through two shared-memory stages
//      filled by bulk copies: exact for any input, only slower.
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
constexpr int kH = kChunk / (4 * kRT);   // float4 per thread per stage (index order: h, warp, lane)
static_assert(kH * kRW == 32, "a stage's (h, warp) segments are scanned by one warp");

constexpr int kRSel = 2048;              // the selection (k <= 2048), ordered through a bitmap
constexpr int kRTies = 256;              // keys equal to the k-th key, ranked by index

struct __align__(128) RowTopkSmem {
  float ring[kStages][kChunk];   // the whole-row path's stages
  uint32_t ckey[kRCand];
  int32_t cidx[kRCand];
  uint32_t hist[kRBins];
  int32_t sel[kRSel];
  int32_t tidx[kRTies];
  uint64_t full[kStages];
  uint32_t seg[kH * kRW];      // per (h, warp) counts of a stage, then their exclusive prefix
  uint32_t seg_total;
  uint32_t bscan[kRW];
  uint32_t nsel, ntie;
  int thr;
  uint32_t above, total, in_thr;
};

constexpr size_t kRowSmem = sizeof(RowTopkSmem) + 128;
static_assert(2 * (kRowSmem + 1024) <= 233472, "two CTAs must fit on an SM");
static_assert(kStages * kChunk * 4 >= kRowMax / 8, "the ordering bitmap fits in the ring");

__device__ __forceinline__ uint32_t row_key(float v) {
  return topk_score_key(v);
}


__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm volatile("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

// Histogram add (kRBins: none) for bins that crowd: the lanes sharing lane
// 0's bin add as one atomic, the others one each.  (Cheaper than grouping
// every distinct bin: __match_any_sync costs several microseconds over a
// row's sample.)  Every lane of the warp calls it.
__device__ __forceinline__ void hist_agg(uint32_t *h, uint32_t bin) {
  const uint32_t b0 = __shfl_sync(0xffffffffu, bin, 0);
  const uint32_t same = __ballot_sync(0xffffffffu, bin == b0);
  if ((threadIdx.x & 31) == 0 && b0 < kRBins) atomicAdd(&h[b0], (uint32_t)__popc(same));
  if (bin != b0 && bin < kRBins) atomicAdd(&h[bin], 1u);
}

// Within-warp exclusive ranks of four flags per lane in (lane, e) order, and
// the warp's count: the lane counts (0..4) by their three bits, one ballot
// each.
__device__ __forceinline__ uint32_t warp_ranks(const bool (&f)[4], uint32_t (&rank)[4]) {
  const uint32_t lt = lanemask_lt();
  const uint32_t c = (uint32_t)f[0] + (uint32_t)f[1] + (uint32_t)f[2] + (uint32_t)f[3];
  const uint32_t m0 = __ballot_sync(0xffffffffu, c & 1u), m1 = __ballot_sync(0xffffffffu, c & 2u),
                 m2 = __ballot_sync(0xffffffffu, c & 4u);
  const uint32_t before = __popc(m0 & lt) + 2 * __popc(m1 & lt) + 4 * __popc(m2 & lt);
  const uint32_t tot = __popc(m0) + 2 * __popc(m1) + 4 * __popc(m2);
  uint32_t own = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    rank[e] = before + own;
    own += f[e] ? 1u : 0u;
  }
  return tot;
}

// Exclusive prefix of the (h, warp) segment counts in (h, warp) order -- the
// index order of a stage -- and their total.  Two CTA barriers.
__device__ __forceinline__ void seg_scan(RowTopkSmem &S, const uint32_t (&c)[kH], uint32_t (&b)[kH],
                                         uint32_t &total) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (lane == 0)
#pragma unroll
    for (int h = 0; h < kH; ++h) S.seg[h * kRW + w] = c[h];
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
#pragma unroll
  for (int h = 0; h < kH; ++h) b[h] = S.seg[h * kRW + w];
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
    S.in_thr = 0;
  }
  __syncthreads();
  if (total > need) {
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int b = bins - 1 - (kPer * tid + j);
      if (b >= 0 && before < need && before + c[j] >= need) {
        S.thr = b;
        S.above = before;
        S.in_thr = c[j];
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
// chunk, keys[h][e] the key at base + 4 (kRT h + tid) + e (0 past n).  `g` is
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
    uint32_t keys[kH][4];
#pragma unroll
    for (int h = 0; h < kH; ++h) {
      const int o = 4 * (kRT * h + tid);
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
    uint32_t keys[kH][4];
#pragma unroll
    for (int h = 0; h < kH; ++h) {
      const uint32_t o = base + 4 * (kRT * h + tid);
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

// Writes the positions sel[0 .. cnt) (distinct, < n <= kRowMax) to out in
// ascending order through a bitmap of the row held in the ring's space: one
// bit per position, then each thread emits the set bits of its own run of
// words at its exclusive prefix of the CTA's counts; out is padded with -1
// to k.  Ends with the CTA synchronised.
template <typename M>
__device__ void write_sorted(RowTopkSmem &S, uint32_t cnt, int64_t n, uint32_t k, int32_t *out, M &&map) {
  constexpr int kPer = (kRowMax / 32 + kRT - 1) / kRT;   // words per thread (8)
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  uint32_t *bm = reinterpret_cast<uint32_t *>(&S.ring[0][0]);
  const int nw = (int)((n + 31) / 32);
  for (int i = tid; i < nw; i += kRT) bm[i] = 0u;
  __syncthreads();
  for (uint32_t i = tid; i < cnt; i += kRT) {
    const int32_t v = S.sel[i];
    atomicOr(&bm[v >> 5], 1u << (v & 31));
  }
  __syncthreads();
  const int w0 = tid * kPer;
  uint32_t word[kPer], loc = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    word[j] = w0 + j < nw ? bm[w0 + j] : 0u;
    loc += __popc(word[j]);
  }
  uint32_t incl = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += x;
  }
  if (lane == 31) S.bscan[w] = incl;
  __syncthreads();
  uint32_t pos = incl - loc;
  for (int i = 0; i < w; ++i) pos += S.bscan[i];
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    uint32_t b = word[j];
    while (b) {
      const int bit = __ffs(b) - 1;
      b &= b - 1;
      if (pos < k) out[pos] = map((int32_t)(32 * (w0 + j) + bit));
      ++pos;
    }
  }
  for (uint32_t i = min(cnt, k) + tid; i < k; i += kRT) out[i] = -1;
  __syncthreads();
}

__global__ void __launch_bounds__(kRT, 2) topk_row_kernel(const TopkRows r) {
  extern __shared__ uint8_t smem_raw[];
  RowTopkSmem &S =
      *reinterpret_cast<RowTopkSmem *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int tid = threadIdx.x;
  const int row = blockIdx.x;
  const float *vals = r.vals + (int64_t)row * r.row_stride;
  const int64_t n = r.row_len;
  const uint32_t k = (uint32_t)r.k;

  if (tid < kStages) mbar_init(&S.full[tid], 1);
  for (int i = tid; i < kRBins; i += kRT) S.hist[i] = 0;
  fence_barrier_init();
  // the scores' producer is complete past here (programmatic launch)
  pdl_wait();
  // the whole row heads for L2 at once (the filter reads it again after the
  // sample levels): one bulk prefetch per chunk
  if (tid == 0)
    for (int64_t c = 0; c * kChunk < n; ++c)
      prefetch_l2_bulk(vals + c * kChunk, (uint32_t)(4 * min((int64_t)kChunk, n - c * kChunk)));
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
  // the second level only when the first level's bin would bring too many
  // candidates (the sample is an eighth of the row)
  if (S.thr >= 0 && 8 * (S.above + S.in_thr) <= (uint32_t)(kRCand * 5 / 8)) {
    t_low = (uint32_t)S.thr << 21;
  } else if (S.thr >= 0) {
    const uint32_t b0 = (uint32_t)S.thr, above0 = S.above;
    sample(1, b0);
    row_threshold(S, need_s - above0, kRBins);
    t_low = S.thr < 0 ? (b0 << 21) : ((b0 << 21) | ((uint32_t)S.thr << 10));
  }

  // ------------------------------------------------------------ 2. filter
  // Coalesced loads straight from the row, eight float4 per thread in
  // flight; the kept positions (a float compare against t_low's smallest
  // score) go to the warp's own segment of a list in the ring's space (the
  // warp keeps its count in a register: no shared atomics), and the
  // segments are then packed, with their keys read again, into the
  // candidate list (in no particular order).
  uint32_t g = 0;   // chunks through the ring so far (the whole-row path)
  constexpr int kSeg = kRCand / kRW;   // entries per warp segment
  static_assert(kRCand * 4 <= kStages * kChunk * 4, "the warp segments fit in the ring");
  int32_t *seg_idx = reinterpret_cast<int32_t *>(&S.ring[0][0]);
  uint32_t ccount;
  {
    const int lane = tid & 31, w = tid >> 5;
    const float f_low = f32_key_floor(t_low);   // the filter compares floats
    const int64_t n4 = n / 4;
    const float4 *v4 = reinterpret_cast<const float4 *>(vals);
    uint32_t wcnt = 0;   // this warp's candidates (the same in every lane)
#pragma unroll 1
    for (int64_t q0 = 0; q0 < n4; q0 += 8 * kRT) {
      float4 v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int64_t q = q0 + tid + (int64_t)j * kRT;
        v[j] = q < n4 ? __ldcg(v4 + q) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
      // this thread's 32 flags as one mask, one warp scan of the counts,
      // then a slot per set bit (the keys are read again when packed)
      uint32_t mask = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        mask |= (v[j].x >= f_low ? 1u : 0u) << (4 * j);
        mask |= (v[j].y >= f_low ? 1u : 0u) << (4 * j + 1);
        mask |= (v[j].z >= f_low ? 1u : 0u) << (4 * j + 2);
        mask |= (v[j].w >= f_low ? 1u : 0u) << (4 * j + 3);
      }
      const uint32_t c = __popc(mask);
      uint32_t incl = c;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t x = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += x;
      }
      uint32_t pos = wcnt + incl - c;
      while (mask) {
        const int bit = __ffs(mask) - 1;
        mask &= mask - 1;
        if (pos < (uint32_t)kSeg)
          seg_idx[w * kSeg + pos] = (int32_t)(4 * (q0 + tid + (int64_t)(bit >> 2) * kRT) + (bit & 3));
        ++pos;
      }
      wcnt += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) S.seg[w] = wcnt;
    __syncthreads();
    uint32_t base = 0, total = 0;
    bool over = false;
    for (int i = 0; i < kRW; ++i) {
      const uint32_t c = S.seg[i];
      base += i < w ? c : 0u;
      total += c;
      over |= c > (uint32_t)kSeg;
    }
    ccount = over ? (uint32_t)kRCand + 1u : total;   // a full segment counts as an overflow
    if (!over)
      for (uint32_t i = lane; i < wcnt; i += 32) {
        const int32_t idx = seg_idx[w * kSeg + i];
        S.ckey[base + i] = row_key(__ldcg(vals + idx));
        S.cidx[base + i] = idx;
      }
  }
  __syncthreads();
  // the list holds every key of the top k when it did not overflow and has
  // at least k keys, or every valid key of the row (t_low = 1)
  const bool from_list = ccount <= (uint32_t)kRCand && (ccount >= k || t_low == 1);

  pdl_release();   // the row is read: the next kernel's CTAs may be dispatched

  // --------------------------------------------------------- 3./4. select
  // T: the k-th largest key; keys above T are taken, and of the keys equal
  // to T the first tie_need in index order.  T = 0 takes every valid key.
  uint32_t T = 0, tie_need = 0;
  {
    uint32_t need = k, prefix = 0;
#pragma unroll 1
    for (int L = 0; L < 3; ++L) {
      auto hist = [&](uint32_t(&keys)[kH][4], int64_t) {
#pragma unroll
        for (int h = 0; h < kH; ++h)
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
  auto map = [&](int32_t v) { return pool ? __ldg(pool + v / BLOCK) * BLOCK + (v & (BLOCK - 1)) : v; };

  // From the list: every key above T, and of the keys equal to T the
  // tie_need lowest indices (ranked here when there are at most kRTies);
  // the selection is then sorted by index.
  bool ordered = !from_list;
  if (from_list) {
    const int lane = tid & 31;
    if (tid == 0) {
      S.nsel = 0;
      S.ntie = 0;
    }
    __syncthreads();
#pragma unroll 1
    for (uint32_t i0 = 0; i0 < ccount; i0 += kRT) {
      const uint32_t i = i0 + tid;
      const uint32_t key = i < ccount ? S.ckey[i] : 0u;
      const bool above = key > T, tie = key == T && key != 0u;
      const uint32_t ma = __ballot_sync(0xffffffffu, above), mt = __ballot_sync(0xffffffffu, tie);
      uint32_t ba = 0, bt = 0;
      if (lane == 0) {
        if (ma) ba = atomicAdd(&S.nsel, (uint32_t)__popc(ma));
        if (mt) bt = atomicAdd(&S.ntie, (uint32_t)__popc(mt));
      }
      ba = __shfl_sync(0xffffffffu, ba, 0);
      bt = __shfl_sync(0xffffffffu, bt, 0);
      const uint32_t lt = lanemask_lt();
      if (above && ba + __popc(ma & lt) < (uint32_t)kRSel) S.sel[ba + __popc(ma & lt)] = S.cidx[i];
      if (tie && bt + __popc(mt & lt) < (uint32_t)kRTies) S.tidx[bt + __popc(mt & lt)] = S.cidx[i];
    }
    __syncthreads();
    const uint32_t ntie = S.ntie;
    if (ntie > (uint32_t)kRTies) {
      ordered = true;   // too many ties to rank here: the ordered pass over the row
    } else {
      if (tid < ntie) {
        const int32_t v = S.tidx[tid];
        uint32_t rank = 0;
        for (uint32_t j = 0; j < ntie; ++j) rank += S.tidx[j] < v ? 1u : 0u;
        if (rank < tie_need) {
          const uint32_t p = atomicAdd(&S.nsel, 1u);
          if (p < (uint32_t)kRSel) S.sel[p] = v;
        }
      }
      __syncthreads();
      write_sorted(S, min(S.nsel, k), n, k, out, map);
    }
  }
  if (!ordered) return;

  // Ordered pass over the row: the keys above T and the first tie_need keys
  // equal to T, written in index order.
  uint32_t sel_before = 0, tie_before = 0;
  auto emit = [&](uint32_t(&keys)[kH][4], int64_t base) {
    bool te[kH][4], any_tie = false;
#pragma unroll
    for (int h = 0; h < kH; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        te[h][e] = keys[h][e] == T && keys[h][e] != 0u;
        any_tie |= te[h][e];
      }
    uint32_t trk[kH][4] = {}, tb[kH] = {}, ttot = 0;
    if (__syncthreads_or(any_tie)) {
      uint32_t tc[kH];
#pragma unroll
      for (int h = 0; h < kH; ++h) tc[h] = warp_ranks(te[h], trk[h]);
      seg_scan(S, tc, tb, ttot);
    }
    bool fl[kH][4];
    uint32_t srk[kH][4], sc[kH];
#pragma unroll
    for (int h = 0; h < kH; ++h) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        fl[h][e] = keys[h][e] > T || (te[h][e] && tie_before + tb[h] + trk[h][e] < tie_need);
      sc[h] = warp_ranks(fl[h], srk[h]);
    }
    uint32_t sb[kH], stot;
    seg_scan(S, sc, sb, stot);
#pragma unroll
    for (int h = 0; h < kH; ++h)
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (fl[h][e]) {
          const uint32_t pos = sel_before + sb[h] + srk[h][e];
          if (pos < k) out[pos] = map((int32_t)(base + 4 * (kRT * h + tid) + e));
        }
    sel_before += stot;
    tie_before += ttot;
  };
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
  err = launch_pdl(topk_row_kernel, dim3((unsigned)r.rows), dim3(kRT), kRowSmem, stream, 0u, r);
  if (err != cudaSuccess) return err;
  ++*launches;
  if (pe.stop) err = record_profile_event(pe.stop, stream);
  return err;
}


namespace {
int g_topk_choice = 0;
}  // namespace

void set_topk_choice(int which) { g_topk_choice = which; }

bool topk_runs_cluster(const TopkRows &r) {
  if (g_topk_choice == 2) return false;   // strict: no fallback
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
    if (r.rows >= 2 * sms) return false;
  }
  return true;
}

cudaError_t launch_topk(const TopkRows &r, cudaStream_t stream, int *launches, bool profiled) {
  if (topk_runs_cluster(r)) return launch_topk_cluster(r, stream, launches, profiled);
  return launch_topk_row(r, stream, launches, profiled);
}

}  // namespace csa2
