// Exact top-K of each indexer score row in one kernel: one thread-block
// cluster per row, radix select across the cluster through distributed
// shared memory, no global scratch (beyond reading, and clearing, the row
// histograms an indexer sweep may hand over).  Used for the index_topk = 512
// selection of the Full and Reindex layers, the HSI pool's top-2048 blocks,
// and prefill blocks of few rows ("DeepSeek-V4.1-Flash - Architecture",
// sections 2 and 3).
//
// Scores become order-preserving 32-bit keys (-inf marks an invalid slot).
// The CTAs of the cluster split the row into contiguous slices; in a round
// each warp covers 1024 consecutive values with 8 coalesced float4 loads in
// flight per thread (a slice of one round stays in registers throughout).
//   1. the low threshold t_low (every key >= t_low is a candidate): with the
//      sweep's histogram of the row (the valid keys counted by their top 12
//      bits), the exact bin where the count from the top reaches k, when the
//      keys down to that bin fit the leader's list; otherwise from a sample,
//      the first of every warp's 8 loads (1/8 of the values), about twice
//      the sample's share of k above it, located to 22 key bits by two
//      histogram levels (the top 11 bits, then the next 11 inside the bin);
//   2. filter: every key >= t_low goes to the CTA's candidate list in shared
//      memory, in index order (warp and CTA prefix sums of per-thread counts
//      give every thread its output slots: no per-key atomics), and then to a
//      block of the leader's (rank 0) list reserved by a remote atomic add;
//   3. when every list fits its slot and together they hold >= k keys, the
//      leader alone finds the exact top k in the gathered list (after a
//      histogram threshold: the keys above the bin are counted and taken, two
//      radix levels rank those in it; else three levels over the list; ties
//      on the full key toward the lower index) and writes them in list
//      order, which is index order;
//   4. otherwise the cluster selects together: exact radix select -- 11, 11
//      and 10 key bits -- on the candidate lists when together they hold >= k
//      keys and none overflowed, else on the whole slices; a level stops early
//      when its threshold bin holds exactly the count still needed; keys equal
//      on all 32 bits are taken toward the lower index (each CTA its quota, in
//      index order, after a cluster prefix of the per-CTA tie counts); each
//      CTA sorts the indices it selected and writes them at its cluster prefix
//      offset (slices are in index order); the last CTA pads with -1.
// Any t_low gives the exact result: the candidates are all keys >= t_low, so
// at least k of them hold the top k, and fewer (or an overflow) go to step 4.
// Selected positions are mapped through the HSI pool for Reindex rows.
// Histograms are exchanged by pushing each CTA's non-zero bins into every
// CTA's cluster total with remote atomic adds; all waiting is at cluster
// barriers, which the hardware co-schedules.
#include "kernels.cuh"

namespace csa2 {

namespace {

constexpr int kThreads = 256;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kThreads;
constexpr int kSelMax = 2048;          // index_topk limit
constexpr int kVec = 8;                // float4 loads per thread per round (32 values)
constexpr int kRound = kThreads * kVec * 4;   // values per CTA per round
constexpr int kCand = 2048;            // per-CTA candidate list
constexpr int kSampleEvery = 8;        // the sample: 1 of every warp's 8 loads
constexpr int kMaxCluster = 16;        // CTAs per row (non-portable cluster size)
constexpr int kGather = 2048;          // the leader's list of the whole row's candidates

struct __align__(16) TopkClusterSmem {
  uint32_t hist[kBins];                // this CTA's histogram of the current level
  uint32_t tot[2][kBins];              // cluster totals, pushed by every CTA
  uint32_t ckey[kCand];
  int32_t cidx[kCand];
  int32_t sel[kSelMax];                // this CTA's selected indices
  uint32_t gkey[kGather];              // leader: every CTA's candidates, a block per CTA
  int32_t gidx[kGather];
  uint32_t cand_base[kMaxCluster];     // where each CTA's block starts in the leader's list
  uint32_t g_used, g_base;             // leader: entries reserved; this CTA: its block
  uint32_t cand_cnt[kMaxCluster];      // per-CTA counts, pushed by the CTAs
  uint32_t tie_cnt[kMaxCluster];
  uint32_t sel_cnt[kMaxCluster];
  uint32_t ccount, n_sel, n_tie;
  uint32_t scan[kThreads / 32];
  uint32_t warp_cnt[kThreads / 32];
  int thr;
  uint32_t above, total, in_thr;
  uint32_t up;                         // leader: candidates above the histogram's threshold bin
  int cross;                           // the sweep's histogram: the thread holding the threshold bin
  uint32_t cross_before;               // and the keys in the bins above its group
};

static_assert(3 * (sizeof(TopkClusterSmem) + 1024 + 16) <= 232448, "three CTAs must fit on an SM");

__device__ __forceinline__ uint32_t score_key(float v) {
  return topk_score_key(v);
}

__device__ __forceinline__ void red_add_remote(uint32_t addr, uint32_t v) {
  asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Level-L predicate and digit.  Level 0: every valid key, bits 31..21.
// Level 1: bits 31..21 equal the prefix, digit 20..10.  Level 2: bits 31..10
// equal the prefix, digit 9..0.
__device__ __forceinline__ bool level_match(uint32_t key, int level, uint32_t prefix) {
  if (!key) return false;
  if (level == 0) return true;
  if (level == 1) return (key >> 21) == prefix;
  return (key >> 10) == prefix;
}

__device__ __forceinline__ uint32_t level_digit(uint32_t key, int level) {
  return level == 0 ? (key >> 21) : level == 1 ? ((key >> 10) & 2047u) : (key & 1023u);
}

// Histogram add of the warp's 32 bins (kBins: none), aggregated over equal
// bins -- for keys that crowd into a few bins (the top 11 key bits of the
// gathered candidates).
__device__ __forceinline__ void hist_add(uint32_t *h, uint32_t bin, int lane) {
  const uint32_t peers = __match_any_sync(0xffffffffu, bin);
  if (bin < kBins && lane == __ffs(peers) - 1) atomicAdd(&h[bin], (uint32_t)__popc(peers));
}

// The lanes sharing lane 0's bin add as one atomic, the others one each --
// for the sample's top bits, spread over many bins, where grouping every
// distinct bin costs more than it saves.
__device__ __forceinline__ void hist_add_lead(uint32_t *h, uint32_t bin, int lane) {
  const uint32_t b0 = __shfl_sync(0xffffffffu, bin, 0);
  const uint32_t same = __ballot_sync(0xffffffffu, bin == b0);
  if (lane == 0 && b0 < kBins) atomicAdd(&h[b0], (uint32_t)__popc(same));
  if (bin != b0 && bin < kBins) atomicAdd(&h[bin], 1u);
}

// The same without aggregation -- for the finer levels, where a warp's bins
// are mostly distinct and the match costs more than it saves.
__device__ __forceinline__ void hist_add_plain(uint32_t *h, uint32_t bin) {
  if (bin < kBins) atomicAdd(&h[bin], 1u);
}

// Appends the flagged indices of this warp to the CTA's selection list.
__device__ __forceinline__ void append_sel(TopkClusterSmem &S, bool flag, int32_t idx, int lane) {
  const uint32_t m = __ballot_sync(0xffffffffu, flag);
  if (!m) return;
  uint32_t base = 0;
  if (lane == 0) base = atomicAdd(&S.n_sel, (uint32_t)__popc(m));
  base = __shfl_sync(0xffffffffu, base, 0);
  if (flag) {
    const uint32_t pos = base + __popc(m & ((1u << lane) - 1));
    if (pos < kSelMax) S.sel[pos] = idx;
  }
}

// Adds this CTA's histogram into tot[buf] of every CTA of the cluster (non-zero
// bins only) and clears it.  Visible everywhere after the next cluster barrier.
__device__ __forceinline__ void push_hist(TopkClusterSmem &S, int buf, uint32_t nctas) {
  for (int b = threadIdx.x; b < kBins; b += kThreads) {
    const uint32_t v = S.hist[b];
    if (v) {
      for (uint32_t c = 0; c < nctas; ++c) red_add_remote(dsmem_addr(&S.tot[buf][b], c), v);
      S.hist[b] = 0;
    }
  }
}

// Threshold of the cluster totals tot[buf] for `need` (bins of the level):
// thr = -1 when everything matching fits.  Clears tot[buf] for its next use.
__device__ void local_threshold(TopkClusterSmem &S, int buf, uint32_t need, int bins) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  uint32_t c[kBinsPerThread], loc = 0;
#pragma unroll
  for (int j = 0; j < kBinsPerThread; ++j) {
    const int b = bins - 1 - (kBinsPerThread * tid + j);
    c[j] = (b >= 0) ? S.tot[buf][b] : 0u;
    loc += c[j];
  }
  uint32_t incl = loc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) S.scan[wid] = incl;
  __syncthreads();
  uint32_t wbase = 0, total = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < wid) wbase += S.scan[w];
    total += S.scan[w];
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
    for (int j = 0; j < kBinsPerThread; ++j) {
      const int b = bins - 1 - (kBinsPerThread * tid + j);
      if (b >= 0 && before < need && before + c[j] >= need) {
        S.thr = b;
        S.above = before;
        S.in_thr = c[j];
      }
      before += c[j];
    }
  }
  for (int b = tid; b < kBins; b += kThreads) S.tot[buf][b] = 0;
  __syncthreads();
}

// One round of a CTA's slice: warp w covers the 1024 consecutive values
// base + 1024 w ..; its load j (coalesced) the 128 values from
// base + 1024 w + 128 j, 4 per lane.  Values past `hi` read as -inf.
__device__ __forceinline__ int64_t round_index(int64_t base, int j) {
  return base + (int64_t)(threadIdx.x >> 5) * (32 * 4 * kVec) + j * 128 + (threadIdx.x & 31) * 4;
}

__device__ __forceinline__ void load_round(const float *vals, int64_t base, int64_t hi, float4 (&v)[kVec]) {
#pragma unroll
  for (int j = 0; j < kVec; ++j) {
    const int64_t i = round_index(base, j);
    v[j] = (i < hi) ? __ldcg(reinterpret_cast<const float4 *>(vals + i))
                    : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
  }
}

// Calls f(key, index) for the keys of this CTA's slice [lo, hi) (multiples of
// 4), 32 per thread per round.
template <typename F>
__device__ __forceinline__ void for_slice(const float *vals, int64_t lo, int64_t hi, F &&f) {
  for (int64_t base = lo; base < hi; base += kRound) {
    float4 v[kVec];
    load_round(vals, base, hi, v);
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const int32_t i0 = (int32_t)round_index(base, j);
      f(score_key(v[j].x), i0);
      f(score_key(v[j].y), i0 + 1);
      f(score_key(v[j].z), i0 + 2);
      f(score_key(v[j].w), i0 + 3);
    }
  }
}

// The sample's histogram of level `lvl` (0: key bits 31..21; 1: bits 20..10
// of the keys whose top bits are b0) into tot[lvl] of every CTA: load 0 of
// every warp of every round, 1/8 of the values (v0, when have_v0: that load
// of a slice of one round, already in registers).  Ends at a cluster barrier.
__device__ __forceinline__ void sample_hist(TopkClusterSmem &S, const float *vals, int64_t lo, int64_t hi,
                                            bool have_v0, float4 v0, int lvl, uint32_t b0, uint32_t nctas) {
  const int lane = threadIdx.x & 31;
  for (int64_t base = lo; base < hi; base += kRound) {
    const int64_t i = round_index(base, 0);
    const float4 v = have_v0 ? v0
                     : (i < hi) ? __ldca(reinterpret_cast<const float4 *>(vals + i))
                                : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
    const float x[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const uint32_t key = score_key(x[e]);
      const uint32_t bin = !key ? (uint32_t)kBins
                           : lvl == 0 ? (key >> 21)
                           : (key >> 21) == b0 ? ((key >> 10) & 2047u) : (uint32_t)kBins;
      if (lvl == 0)
        hist_add_lead(S.hist, bin, lane);
      else
        hist_add_plain(S.hist, bin);
    }
  }
  __syncthreads();
  push_hist(S, lvl, nctas);
  cluster_sync();
}

// Exclusive prefix sum of one value per thread over the CTA; *total gets the
// sum.  Uses S.scan; ends with the CTA synchronised.
__device__ __forceinline__ uint32_t block_excl_scan(TopkClusterSmem &S, uint32_t v, uint32_t *total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) S.scan[wid] = incl;
  __syncthreads();
  uint32_t before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const uint32_t x = S.scan[w];
    before += w < wid ? x : 0u;
    tot += x;
  }
  __syncthreads();   // S.scan may be reused
  *total = tot;
  return before + incl - v;
}

// Threshold of the row's histogram from the sweep (h: TOPK_HIST_BINS counts)
// for `need` keys: S.thr = the bin where the count from the top reaches
// need, or -1 when the row holds no more than need valid keys; S.above = the
// keys in the bins above it, S.in_thr = the keys in it.  Thread t sums the
// t-th group of TOPK_HIST_BINS / 256 bins from the top; the warp of the group
// that holds the crossing reads that group again, a bin per lane.  Ends
// synchronised.
__device__ void hist_threshold(TopkClusterSmem &S, const uint32_t *h, uint32_t need) {
  constexpr int kPer = TOPK_HIST_BINS / kThreads;
  static_assert(kPer % 4 == 0 && kPer <= 32, "whole uint4 groups, at most one bin per lane in the second read");
  const int tid = threadIdx.x, lane = tid & 31;
  const uint4 *g = reinterpret_cast<const uint4 *>(h + TOPK_HIST_BINS - kPer * (tid + 1));
  uint32_t loc = 0;
#pragma unroll
  for (int j = 0; j < kPer / 4; ++j) {
    const uint4 x = __ldcg(g + j);
    loc += x.x + x.y + x.z + x.w;
  }
  uint32_t total;
  const uint32_t before = block_excl_scan(S, loc, &total);
  if (tid == 0) {
    S.thr = -1;
    S.above = total;
    S.in_thr = 0;
    S.total = total;
  }
  if (total > need && before < need && before + loc >= need) {
    S.cross = tid;
    S.cross_before = before;
  }
  __syncthreads();
  if (total > need && (tid >> 5) == (S.cross >> 5)) {
    const int t = S.cross;
    const int bin = TOPK_HIST_BINS - 1 - kPer * t - lane;   // lane 0 the group's top bin
    const uint32_t c = lane < kPer ? __ldcg(h + bin) : 0u;
    uint32_t incl = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    const uint32_t above = S.cross_before + incl - c;
    if (lane < kPer && above < need && above + c >= need) {
      S.thr = bin;
      S.above = above;
      S.in_thr = c;
    }
  }
  __syncthreads();
}

// Calls f(key, index) for the CTA's candidate list; uniform trip count.
template <typename F>
__device__ __forceinline__ void for_cands(TopkClusterSmem &S, F &&f) {
  const int n = (int)min(S.ccount, (uint32_t)kCand);
  for (int b0 = 0; b0 < n; b0 += kThreads) {
    const int i = b0 + threadIdx.x;
    f(i < n ? S.ckey[i] : 0u, i < n ? S.cidx[i] : -1);
  }
}

// The radix levels; tot[0] holds the cluster's level-0 histogram on entry.
// Returns the count still needed (full-key ties) and the tie key in *full.
template <bool kCands>
__device__ uint32_t run_levels(TopkClusterSmem &S, const TopkRows &r, const float *vals, int64_t lo, int64_t hi,
                               uint32_t nctas, uint32_t *full) {
  const int lane = threadIdx.x & 31;
  local_threshold(S, 0, (uint32_t)r.k, kBins);
  uint32_t need = S.total < (uint32_t)r.k ? S.total : (uint32_t)r.k;
  int level = 0, buf = 0;
  uint32_t prefix = 0;
  while (true) {
    const int thr = S.thr;
    const uint32_t above = S.above, in_thr = S.in_thr;
    // the threshold bin is taken whole when it holds exactly the count still
    // needed (or when everything matching fits: thr = -1)
    const bool take_thr = thr < 0 || above + in_thr == need;
    const bool last = take_thr || level == 2;
    auto body = [&](uint32_t key, int32_t idx) {
      const bool m = level_match(key, level, prefix);
      const int d = m ? (int)level_digit(key, level) : -1;
      // most keys are below the threshold bin: skip the warp unless a lane has work
      if (!__any_sync(0xffffffffu, m && d >= thr)) return;
      append_sel(S, m && (d > thr || (take_thr && d == thr)), idx, lane);
      if (!last) hist_add(S.hist, (m && d == thr) ? level_digit(key, level + 1) : (uint32_t)kBins, lane);
    };
    if (kCands) for_cands(S, body);
    else for_slice(vals, lo, hi, body);
    if (last) {
      if (take_thr) {
        need = 0;
      } else {
        need -= above;
        prefix = (prefix << 10) | (uint32_t)thr;   // the full 32-bit key of the ties
      }
      break;
    }
    __syncthreads();
    push_hist(S, buf ^ 1, nctas);
    cluster_sync();   // every CTA's next-level histogram has been added everywhere
    need -= above;
    prefix = (level == 0) ? (uint32_t)thr : ((prefix << 11) | (uint32_t)thr);
    ++level;
    buf ^= 1;
    local_threshold(S, buf, need, level == 2 ? 1024 : kBins);
  }
  *full = prefix;
  return need;
}

// The leader's exact top-k of its row from the candidates every CTA pushed
// into its gather list (CTA c's block: cand_cnt[c] entries at cand_base[c],
// in index order; the CTAs' slices are in index order too).  The blocks are
// compacted in CTA order into
// one list, three radix levels over local histograms (11, 11 and 10 key
// bits) locate the full key T of the k-th largest, and the keys above T plus
// the lowest-index keys equal to T are written ascending (list order).
__device__ void leader_select(TopkClusterSmem &S, const TopkRows &r, int row, uint32_t nctas, int hb) {
  const uint32_t tid = threadIdx.x;
  uint32_t n = 0;
#pragma unroll 1
  for (uint32_t c = 0; c < nctas; ++c) {
    const uint32_t m = S.cand_cnt[c], b = S.cand_base[c];
#pragma unroll 1
    for (uint32_t i = tid; i < m; i += kThreads) {
      S.ckey[n + i] = S.gkey[b + i];
      S.cidx[n + i] = S.gidx[b + i];
    }
    n += m;
  }
  __syncthreads();
  uint32_t need = (uint32_t)r.k, prefix = 0;   // k <= n: checked by the caller
  // hb >= 0: every candidate's top TOPK_HIST_BITS key bits are >= hb (the
  // sweep's threshold bin): the keys above that bin, counted here, are all
  // taken, and two levels on the remaining bits rank the keys in it.  Otherwise (or if
  // the count says the bin cannot hold the k-th key) three levels of 11, 11
  // and 10 bits over the whole list.
  bool hm = false;
  if (hb >= 0) {
    if (tid == 0) S.up = 0u;
    __syncthreads();
#pragma unroll 1
    for (uint32_t b0 = 0; b0 < n; b0 += kThreads) {
      const uint32_t i = b0 + tid;
      const bool up = i < n && (S.ckey[i] >> (32 - TOPK_HIST_BITS)) > (uint32_t)hb;
      const uint32_t c = __popc(__ballot_sync(0xffffffffu, up));
      if ((tid & 31) == 0 && c) atomicAdd(&S.up, c);
    }
    __syncthreads();
    const uint32_t up = S.up;
    if (up < need) {
      hm = true;
      need -= up;
      prefix = (uint32_t)hb;
    }
  }
  const int levels = hm ? 2 : 3;
#pragma unroll 1
  for (int L = 0; L < levels; ++L) {
    // below the histogram's bits: a level on the upper half, one on the lower
    constexpr int kRest = 32 - TOPK_HIST_BITS, kLow = kRest / 2;
    static_assert(kRest - kLow <= 11 && kLow >= 8, "level widths within the bins, per-thread groups whole");
    const int sh = hm ? (L == 0 ? kLow : 0) : (L == 0 ? 21 : L == 1 ? 10 : 0);
    const int width = hm ? (L == 0 ? kRest - kLow : kLow) : (L == 2 ? 10 : 11);
    const uint32_t nb = 1u << width;
    for (int b = tid; b < kBins; b += kThreads) S.hist[b] = 0;
    __syncthreads();
    // the top 11 bits: warp-aggregated adds (the candidates crowd into a few
    // bins); below them the bins are mostly distinct
#pragma unroll 1
    for (uint32_t b0 = 0; b0 < n; b0 += kThreads) {
      const uint32_t i = b0 + tid;
      const uint32_t key = i < n ? S.ckey[i] : 0u;
      const bool m = i < n && ((L == 0 && !hm) || (key >> (sh + width)) == prefix);
      const uint32_t bin = m ? ((key >> sh) & (nb - 1)) : (uint32_t)kBins;
      if (L == 0 && !hm)
        hist_add(S.hist, bin, tid & 31);
      else
        hist_add_plain(S.hist, bin);
    }
    __syncthreads();
    // bins from the top, nb / kThreads per thread: the one where the count reaches `need`
    const int per = (int)nb / kThreads;
    uint32_t cnt[kBinsPerThread], loc = 0;
#pragma unroll
    for (int j = 0; j < kBinsPerThread; ++j) {
      cnt[j] = j < per ? S.hist[nb - 1 - (per * tid + j)] : 0u;
      loc += cnt[j];
    }
    uint32_t tot;
    uint32_t before = block_excl_scan(S, loc, &tot);
#pragma unroll
    for (int j = 0; j < kBinsPerThread; ++j) {
      if (j < per && before < need && before + cnt[j] >= need) {
        S.thr = (int)(nb - 1 - (per * tid + j));
        S.above = before;
      }
      before += cnt[j];
    }
    __syncthreads();
    need -= S.above;
    prefix = (prefix << width) | (uint32_t)S.thr;
    __syncthreads();   // S.thr and S.above are read before the next level sets them
  }
  // prefix is T; the `need` lowest-index keys equal to T are taken
  const uint32_t T = prefix;
  const uint32_t per = (n + kThreads - 1) / kThreads;   // a contiguous run of the list per thread
  const uint32_t i0 = min(tid * per, n), i1 = min(i0 + per, n);
  uint32_t eq = 0;
#pragma unroll 1
  for (uint32_t i = i0; i < i1; ++i) eq += S.ckey[i] == T;
  uint32_t tot_eq, tot_sel;
  const uint32_t eq_before = block_excl_scan(S, eq, &tot_eq);
  uint32_t nsel = 0, e = eq_before;
#pragma unroll 1
  for (uint32_t i = i0; i < i1; ++i) {
    const uint32_t key = S.ckey[i];
    nsel += key > T || (key == T && e < need);
    e += key == T;
  }
  uint32_t o = block_excl_scan(S, nsel, &tot_sel);
  int32_t *out = r.out + (int64_t)row * r.k;
  e = eq_before;
#pragma unroll 1
  for (uint32_t i = i0; i < i1; ++i) {
    const uint32_t key = S.ckey[i];
    const bool f = key > T || (key == T && e < need);
    e += key == T;
    if (!f) continue;
    const int32_t v = S.cidx[i];
    int32_t pos = v;
    if (r.pool) {
      const int32_t blk = __ldg(r.pool + (int64_t)row * r.pool_stride + v / BLOCK);
      pos = blk * BLOCK + (v & (BLOCK - 1));
    }
    if (o < (uint32_t)r.k) out[o] = pos;
    ++o;
  }
}

// The cluster's exact selection when the leader could not take the whole
// row (steps 3 and 4 of the outline at the top of this file).
__device__ __forceinline__ void select_together(TopkClusterSmem &S, const TopkRows &r, const float *vals, int64_t lo,
                                                int64_t hi, int row, uint32_t crank, uint32_t nctas,
                                                uint32_t total_cand, bool overflow) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  // 3. exact select, on the candidate lists when they are complete
  uint32_t need, full = 0;
  const bool fast = !overflow && total_cand >= (uint32_t)r.k;
  if (fast)
    for_cands(S, [&](uint32_t key, int32_t) { hist_add(S.hist, key ? (key >> 21) : (uint32_t)kBins, lane); });
  else
    for_slice(vals, lo, hi,
              [&](uint32_t key, int32_t) { hist_add(S.hist, key ? (key >> 21) : (uint32_t)kBins, lane); });
  __syncthreads();
  push_hist(S, 0, nctas);
  cluster_sync();
  need = fast ? run_levels<true>(S, r, vals, lo, hi, nctas, &full)
              : run_levels<false>(S, r, vals, lo, hi, nctas, &full);

  if (need > 0) {
    // ties on the full key: the `need` lowest indices, CTA slices in order
    for_slice(vals, lo, hi, [&](uint32_t key, int32_t) {
      const uint32_t tm = __ballot_sync(0xffffffffu, key == full);
      if (lane == 0 && tm) atomicAdd(&S.n_tie, (uint32_t)__popc(tm));
    });
    __syncthreads();
    if (tid < (int)nctas) dsmem_st_u32(dsmem_addr(&S.tie_cnt[crank], (uint32_t)tid), S.n_tie);
    cluster_sync();
    uint32_t before = 0;
    for (uint32_t c = 0; c < crank; ++c) before += S.tie_cnt[c];
    const uint32_t quota = need > before ? min(need - before, S.n_tie) : 0u;
    uint32_t running = 0;
    for (int64_t base = lo; base < hi && running < quota; base += kThreads) {
      const int64_t i = base + tid;
      const bool f = i < hi && score_key(__ldcg(vals + i)) == full;
      const uint32_t m = __ballot_sync(0xffffffffu, f);
      if (lane == 0) S.warp_cnt[wid] = __popc(m);
      __syncthreads();
      uint32_t wb = 0, tot = 0;
      for (int w = 0; w < kThreads / 32; ++w) {
        if (w < wid) wb += S.warp_cnt[w];
        tot += S.warp_cnt[w];
      }
      const uint32_t rank = running + wb + __popc(m & ((1u << lane) - 1));
      append_sel(S, f && rank < quota, (int32_t)i, lane);
      running += tot;
      __syncthreads();
    }
  }

  // 4. every CTA writes its sorted selections at its cluster prefix offset
  __syncthreads();
  const uint32_t mine = min(S.n_sel, (uint32_t)kSelMax);
  if (tid < (int)nctas) dsmem_st_u32(dsmem_addr(&S.sel_cnt[crank], (uint32_t)tid), mine);
  cluster_sync();   // the last remote access: afterwards every CTA works on its own memory
  uint32_t off = 0, all = 0;
  for (uint32_t c = 0; c < nctas; ++c) {
    if (c < crank) off += S.sel_cnt[c];
    all += S.sel_cnt[c];
  }
  int32_t *out = r.out + (int64_t)row * r.k;
  for (uint32_t i = tid; i < mine; i += kThreads) {
    const int32_t v = S.sel[i];
    uint32_t rank = 0;
    for (uint32_t j = 0; j < mine; ++j) rank += S.sel[j] < v;
    int32_t pos = v;
    if (r.pool) {
      const int32_t blk = __ldg(r.pool + (int64_t)row * r.pool_stride + v / BLOCK);
      pos = blk * BLOCK + (v & (BLOCK - 1));
    }
    if (off + rank < (uint32_t)r.k) out[off + rank] = pos;
  }
  if (crank == nctas - 1)
    for (int i = (int)min(all, (uint32_t)r.k) + tid; i < r.k; i += kThreads) out[i] = -1;
}

__global__ void __launch_bounds__(kThreads, 2) topk_cluster_kernel(const TopkRows r) {
  extern __shared__ uint8_t smem_raw[];
  TopkClusterSmem &S = *reinterpret_cast<TopkClusterSmem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const uint32_t crank = cluster_ctarank(), nctas = cluster_nctarank();
  const int row = blockIdx.y;
  const float *vals = r.vals + (int64_t)row * r.row_stride;
  const int64_t n4 = r.row_len / 4;
  const int64_t lo = 4 * (n4 * crank / nctas), hi = 4 * (n4 * (crank + 1) / nctas);
  // a slice of one round stays in registers from here: the sample and the
  // filter read it there
  const bool one_round = hi - lo <= kRound;
  for (int i = tid; i < kBins; i += kThreads) {
    S.hist[i] = 0;
    S.tot[0][i] = 0;
    S.tot[1][i] = 0;
  }
  if (tid < kMaxCluster) {
    S.cand_cnt[tid] = 0;
    S.tie_cnt[tid] = 0;
    S.sel_cnt[tid] = 0;
  }
  if (tid == 0) {
    S.ccount = 0;
    S.n_sel = 0;
    S.n_tie = 0;
    S.g_used = 0;
  }
  // every CTA's totals and counters are cleared before anyone adds to them
  // remotely: a cluster barrier, awaited before the first remote add
  cluster_arrive();
  // the scores' producer is complete past here (programmatic launch)
  pdl_wait();
  float4 vr[kVec];
  if (one_round) {
    load_round(vals, lo, hi, vr);
  } else if (tid == 0) {
    // a longer slice is read three times (two sample levels, the filter):
    // bring all of it into L2 now, one round (32 KB) per bulk prefetch
    for (int64_t b = lo; b < hi; b += kRound)
      prefetch_l2_bulk(vals + b, (uint32_t)(4 * (hi - b < kRound ? hi - b : kRound)));
  }

  // 1. the low threshold t_low: every key >= t_low is a candidate.  From the
  // sweep's histogram of the row when it has one and the keys down to the
  // bin where the count reaches k fit the leader's list (exact counts: no
  // sampling); otherwise from a sample of load 0 of every warp of every
  // round, 1/8 of the values, about twice the sample's share of k above it,
  // located to 22 key bits: the level-0 bin, then the level-1 bin inside it
  uint32_t t_low = 1u;
  bool sample = true;
  int hbin = -1;   // the histogram's threshold bin when t_low comes from it
  if (r.hist) {
    hist_threshold(S, r.hist + (int64_t)row * TOPK_HIST_BINS, (uint32_t)r.k);
    if (S.thr < 0) {
      sample = false;   // every valid key
    } else if (S.above + S.in_thr <= (uint32_t)kGather) {
      sample = false;
      hbin = S.thr;
      t_low = max((uint32_t)S.thr << (32 - TOPK_HIST_BITS), 1u);
    }
  }
  cluster_wait();
  if (sample) {
    const uint32_t need_s = (uint32_t)(2 * r.k / kSampleEvery) + 16;
    sample_hist(S, vals, lo, hi, one_round, vr[0], 0, 0u, nctas);
    local_threshold(S, 0, need_s, kBins);
    if (S.thr >= 0) {
      const uint32_t b0 = (uint32_t)S.thr, above0 = S.above;
      sample_hist(S, vals, lo, hi, one_round, vr[0], 1, b0, nctas);
      local_threshold(S, 1, need_s - above0, kBins);
      t_low = S.thr < 0 ? (b0 << 21) : ((b0 << 21) | ((uint32_t)S.thr << 10));
    }
  }

  // 2. filter into the candidate list, in index order.  Within a warp the
  // order is (load j, lane, component): the per-lane counts of the 8 loads
  // are packed into two words of 8-bit fields (a field sums to at most 128)
  // and prefix-summed across the warp at once; warps are in index order, and
  // a CTA prefix sum of the warp totals places them.
  uint32_t n_cand = 0;
  const float f_low = f32_key_floor(t_low);   // keys >= t_low <=> values >= f_low
  for (int64_t base = lo; base < hi; base += kRound) {
    float4 v[kVec];
    if (one_round) {
#pragma unroll
      for (int j = 0; j < kVec; ++j) v[j] = vr[j];
    } else {
      load_round(vals, base, hi, v);
    }
    uint32_t pk[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const uint32_t c = (v[j].x >= f_low) + (v[j].y >= f_low) + (v[j].z >= f_low) + (v[j].w >= f_low);
      pk[j >> 2] |= c << (8 * (j & 3));
    }
    uint32_t inc[2] = {pk[0], pk[1]};
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n0 = __shfl_up_sync(0xffffffffu, inc[0], o), n1 = __shfl_up_sync(0xffffffffu, inc[1], o);
      if (lane >= o) {
        inc[0] += n0;
        inc[1] += n1;
      }
    }
    const uint32_t tw0 = __shfl_sync(0xffffffffu, inc[0], 31), tw1 = __shfl_sync(0xffffffffu, inc[1], 31);
    uint32_t wtot = 0, jbase[kVec];   // warp-local start of load j's candidates
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      jbase[j] = wtot;
      wtot += ((j < 4 ? tw0 : tw1) >> (8 * (j & 3))) & 0xFFu;
    }
    uint32_t tot;
    const uint32_t wbase = n_cand + block_excl_scan(S, lane == 0 ? wtot : 0u, &tot);
    const uint32_t wb = __shfl_sync(0xffffffffu, wbase, 0);
#pragma unroll
    for (int j = 0; j < kVec; ++j) {
      const uint32_t ex = (((j < 4 ? inc[0] - pk[0] : inc[1] - pk[1]) >> (8 * (j & 3))) & 0xFFu);
      uint32_t pos = wb + jbase[j] + ex;
      const int32_t i0 = (int32_t)round_index(base, j);
      const float x[4] = {v[j].x, v[j].y, v[j].z, v[j].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        if (x[e] >= f_low) {
          if (pos < kCand) {
            S.ckey[pos] = score_key(x[e]);
            S.cidx[pos] = i0 + e;
          }
          ++pos;
        }
      }
    }
    n_cand += tot;
  }
  if (tid == 0) S.ccount = n_cand;
  __syncthreads();
  // every CTA copies its candidates into a block of the leader's (rank 0)
  // list, reserved by a remote atomic add; the blocks' places go to every CTA
  const uint32_t mine_c = min(n_cand, (uint32_t)kCand);
  if (tid == 0) S.g_base = dsmem_atom_add(dsmem_addr(&S.g_used, 0u), mine_c);
  __syncthreads();
  const uint32_t gb = S.g_base;
  if (gb + mine_c <= (uint32_t)kGather)
    for (uint32_t i = tid; i < mine_c; i += kThreads) {
      dsmem_st_u32(dsmem_addr(&S.gkey[gb + i], 0u), S.ckey[i]);
      dsmem_st_u32(dsmem_addr(&S.gidx[gb + i], 0u), (uint32_t)S.cidx[i]);
    }
  if (tid < (int)nctas) {
    dsmem_st_u32(dsmem_addr(&S.cand_cnt[crank], (uint32_t)tid), S.ccount);
    dsmem_st_u32(dsmem_addr(&S.cand_base[crank], (uint32_t)tid), gb);
  }
  cluster_sync();
  if (r.hist) {
    // every CTA has read the row's histogram: clear it for the next call,
    // a slice per CTA
    uint32_t *h = r.hist + (int64_t)row * TOPK_HIST_BINS;
    for (uint32_t i = crank * TOPK_HIST_BINS / nctas + tid; i < (crank + 1) * TOPK_HIST_BINS / nctas; i += kThreads)
      h[i] = 0u;
  }
  uint32_t total_cand = 0;
  bool overflow = false;
  for (uint32_t c = 0; c < nctas; ++c) {
    total_cand += S.cand_cnt[c];
    overflow |= S.cand_cnt[c] > (uint32_t)kCand;
  }
  if (!overflow && total_cand >= (uint32_t)r.k && total_cand <= (uint32_t)kGather) {
    // every candidate is in the leader, which selects alone; the other CTAs
    // are done (nothing reads their memory any more)
    if (crank == 0) {
      pdl_release();   // the next kernel's CTAs may take the SMs the others leave
      leader_select(S, r, row, nctas, hbin);
    }
    return;
  }

  select_together(S, r, vals, lo, hi, row, crank, nctas, total_cand, overflow);
}

}  // namespace

bool topk_cluster_supported(const TopkRows &r) {
  return r.k <= kSelMax && r.row_len % 4 == 0 && r.row_stride % 4 == 0 &&
         (reinterpret_cast<uintptr_t>(r.vals) & 15u) == 0;
}

cudaError_t launch_topk_cluster(const TopkRows &r, cudaStream_t stream, int *launches, bool profiled) {
  if (r.rows <= 0) return cudaSuccess;
  if (!topk_cluster_supported(r)) return cudaErrorInvalidValue;
  static int max_cluster = 0;
  if (!max_cluster) {
    max_cluster = 8;
    if (cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess)
      max_cluster = kMaxCluster;
    else
      (void)cudaGetLastError();
  }
  const size_t smem = sizeof(TopkClusterSmem) + 16;
  cudaError_t err = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  // CTAs per row: one per 8192 scores (a single round each) when there are
  // few rows -- latency; fewer when the rows alone fill the GPU (3 CTAs fit
  // on an SM) -- throughput.
  int dev = 0, sms = 0;
  err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  int64_t c = (r.row_len + 8191) / 8192;
  if (c > max_cluster) c = max_cluster;
  const int64_t fill = 3 * (int64_t)sms / r.rows;   // three CTAs fit on an SM
  if (c > fill) c = fill;
  if (c < 1) c = 1;
  static const ProfileEvents kNone;
  const ProfileEvents &pe = profiled ? profile_events(CSA2_KERNEL_TOPK) : kNone;
  if (pe.start && (err = record_profile_event(pe.start, stream)) != cudaSuccess) return err;
  err = launch_pdl(topk_cluster_kernel, dim3((unsigned)c, (unsigned)r.rows), dim3(kThreads), smem, stream,
                   (unsigned)c, r);
  if (err != cudaSuccess) return err;
  ++*launches;
  if (pe.stop) err = record_profile_event(pe.stop, stream);
  return err;
}

}  // namespace csa2
