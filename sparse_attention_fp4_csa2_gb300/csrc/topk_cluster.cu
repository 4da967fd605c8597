// Exact top-K of each indexer score row in one kernel: one thread-block
// cluster per row, radix select across the cluster through distributed
// shared memory, no global scratch.  Used for the index_topk = 512 selection
// of the Full and Reindex layers ("DeepSeek-V4.1-Flash - Architecture",
// sections 2 and 3).
//
// Scores become order-preserving 32-bit keys (-inf marks an invalid slot).
// The CTAs of the cluster split the row into contiguous slices.  Level 0
// histograms the top 11 key bits; every CTA sums the cluster's histograms
// over DSMEM and finds the same threshold bin; keys above it are selected,
// keys in it go on to level 1 (next 11 bits) and level 2 (last 10 bits).  A
// level stops early when its threshold bin holds exactly the count still
// needed.  Keys equal on all 32 bits are resolved toward the lower index: each
// CTA takes its quota of them in index order after a cluster prefix of the
// per-CTA counts.  Selected indices are appended to CTA 0's list; CTA 0 maps
// them to positions (through the HSI pool for Reindex rows), sorts them
// ascending and writes them, -1 padded.  Each level re-reads the slice (from
// L2: the sweep has just written it); no CTA waits on another except at
// cluster barriers, which the hardware co-schedules.
#include "kernels.cuh"

namespace csa2 {

namespace {

constexpr int kThreads = 512;
constexpr int kBins = 2048;
constexpr int kSelMax = 2048;     // index_topk limit
constexpr int kPer = 8;           // values per thread per sweep of a slice segment

struct __align__(16) TopkClusterSmem {
  uint32_t hist[2][kBins];
  uint32_t tot[kBins];
  int32_t sel[kSelMax];
  uint32_t n_sel;
  uint32_t tie_cnt;
  uint32_t warp_cnt[kThreads / 32];
  uint32_t scan[kThreads / 32];
  int thr;
  uint32_t above;
  uint32_t total;
  uint32_t in_thr;
};

__device__ __forceinline__ uint32_t score_key(float v) {
  return (v == -INFINITY || v != v) ? 0u : f32_key(v);
}

// Matching predicate and digit of a level.  Level 0: every valid key, digit =
// bits 31..21.  Level 1: keys whose bits 31..21 equal the prefix, digit =
// bits 20..10.  Level 2: bits 31..10 equal the prefix, digit = bits 9..0.
__device__ __forceinline__ bool level_match(uint32_t key, int level, uint32_t prefix) {
  if (!key) return false;
  if (level == 0) return true;
  if (level == 1) return (key >> 21) == prefix;
  return (key >> 10) == prefix;
}

__device__ __forceinline__ uint32_t level_digit(uint32_t key, int level) {
  return level == 0 ? (key >> 21) : level == 1 ? ((key >> 10) & 2047u) : (key & 1023u);
}

// Appends the flagged indices of this warp to CTA 0's selection list.
__device__ __forceinline__ void append_sel(bool flag, int32_t idx, uint32_t nsel_addr0, uint32_t sel_addr0,
                                           int lane) {
  const uint32_t m = __ballot_sync(0xffffffffu, flag);
  if (!m) return;
  uint32_t base = 0;
  if (lane == 0) base = dsmem_atom_add(nsel_addr0, (uint32_t)__popc(m));
  base = __shfl_sync(0xffffffffu, base, 0);
  if (flag) {
    const uint32_t pos = base + __popc(m & ((1u << lane) - 1));
    if (pos < kSelMax) dsmem_st_u32(sel_addr0 + 4 * pos, (uint32_t)idx);
  }
}

// Sums the cluster's level histograms into tot (every CTA does it), then
// finds the threshold bin for `need`: thr = -1 when everything matching fits.
__device__ void cluster_threshold(TopkClusterSmem &S, int buf, uint32_t nctas, uint32_t need, int bins) {
  const int tid = threadIdx.x;
  for (int b4 = tid; b4 < kBins / 4; b4 += kThreads) {
    uint4 acc = make_uint4(0, 0, 0, 0);
    for (uint32_t c = 0; c < nctas; ++c) {
      const uint4 v = dsmem_ld_v4(dsmem_addr(&S.hist[buf][4 * b4], c));
      acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    *reinterpret_cast<uint4 *>(&S.tot[4 * b4]) = acc;
  }
  __syncthreads();
  // descending scan: thread t owns bins [bins-1-4t, bins-4-4t]
  const int lane = tid & 31, wid = tid >> 5;
  uint32_t c4[4], loc = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int b = bins - 1 - (4 * tid + j);
    c4[j] = (b >= 0) ? S.tot[b] : 0u;
    loc += c4[j];
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
    for (int j = 0; j < 4; ++j) {
      const int b = bins - 1 - (4 * tid + j);
      if (b >= 0 && before < need && before + c4[j] >= need) {
        S.thr = b;
        S.above = before;
        S.in_thr = c4[j];
      }
      before += c4[j];
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) topk_cluster_kernel(const TopkRows r) {
  extern __shared__ uint8_t smem_raw[];
  TopkClusterSmem &S = *reinterpret_cast<TopkClusterSmem *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 15) & ~uintptr_t(15));
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const uint32_t crank = cluster_ctarank(), nctas = cluster_nctarank();
  const int row = blockIdx.y;
  const float *vals = r.vals + (int64_t)row * r.row_stride;
  const int64_t lo = r.row_len * crank / nctas, hi = r.row_len * (crank + 1) / nctas;
  const uint32_t nsel0 = dsmem_addr(&S.n_sel, 0), sel0 = dsmem_addr(&S.sel[0], 0);

  for (int i = tid; i < kBins; i += kThreads) S.hist[0][i] = 0;
  if (tid == 0) {
    S.n_sel = 0;
    S.tie_cnt = 0;
  }
  __syncthreads();

  // level-0 histogram of this slice
  for (int64_t base = lo; base < hi; base += (int64_t)kThreads * kPer) {
    float v[kPer];
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int64_t i = base + j * kThreads + tid;
      v[j] = (i < hi) ? vals[i] : -INFINITY;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const uint32_t key = score_key(v[j]);
      const uint32_t bin = key ? (key >> 21) : (uint32_t)kBins;
      const uint32_t peers = __match_any_sync(0xffffffffu, bin);
      if (bin < kBins && lane == __ffs(peers) - 1) atomicAdd(&S.hist[0][bin], (uint32_t)__popc(peers));
    }
  }
  cluster_sync();

  cluster_threshold(S, 0, nctas, (uint32_t)r.k, kBins);
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
    const int nbuf = buf ^ 1;
    if (!last)
      for (int i = tid; i < kBins; i += kThreads) S.hist[nbuf][i] = 0;
    __syncthreads();
    for (int64_t base = lo; base < hi; base += (int64_t)kThreads * kPer) {
      float v[kPer];
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int64_t i = base + j * kThreads + tid;
        v[j] = (i < hi) ? vals[i] : -INFINITY;
      }
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int64_t i = base + j * kThreads + tid;
        const uint32_t key = score_key(v[j]);
        const bool m = level_match(key, level, prefix);
        const int d = m ? (int)level_digit(key, level) : -1;
        // most keys are below the threshold bin: skip the warp unless a lane
        // has work (selection, next-level histogram or tie count)
        if (!__any_sync(0xffffffffu, m && d >= thr)) continue;
        append_sel(m && (d > thr || (take_thr && d == thr)), (int32_t)i, nsel0, sel0, lane);
        if (!last) {
          const uint32_t nbin = (m && d == thr) ? level_digit(key, level + 1) : (uint32_t)kBins;
          const uint32_t peers = __match_any_sync(0xffffffffu, nbin);
          if (nbin < kBins && lane == __ffs(peers) - 1) atomicAdd(&S.hist[nbuf][nbin], (uint32_t)__popc(peers));
        } else if (level == 2 && !take_thr) {
          // keys equal on all 32 bits: counted here, resolved by index below
          const uint32_t tm = __ballot_sync(0xffffffffu, m && d == thr);
          if (lane == 0 && tm) atomicAdd(&S.tie_cnt, (uint32_t)__popc(tm));
        }
      }
    }
    if (last) {
      if (take_thr) {
        need = 0;
      } else {
        need -= above;
        prefix = (prefix << 10) | (uint32_t)thr;   // the full 32-bit key of the ties
      }
      break;
    }
    cluster_sync();   // every CTA's next-level histogram is complete
    need -= above;
    prefix = (level == 0) ? (uint32_t)thr : ((prefix << 11) | (uint32_t)thr);
    ++level;
    buf = nbuf;
    cluster_threshold(S, buf, nctas, need, level == 2 ? 1024 : kBins);
  }

  if (need > 0) {
    // ties on the full key: the `need` lowest indices, CTA slices in order
    const uint32_t full = prefix;   // 32-bit key
    __syncthreads();
    cluster_sync();
    uint32_t before = 0;
    for (uint32_t c = 0; c < crank; ++c) before += dsmem_ld_u32(dsmem_addr(&S.tie_cnt, c));
    const uint32_t quota = need > before ? min(need - before, S.tie_cnt) : 0u;
    uint32_t running = 0;
    for (int64_t base = lo; base < hi && running < quota; base += kThreads) {
      const int64_t i = base + tid;
      const bool f = i < hi && score_key(vals[i]) == full;
      const uint32_t m = __ballot_sync(0xffffffffu, f);
      if (lane == 0) S.warp_cnt[wid] = __popc(m);
      __syncthreads();
      uint32_t wb = 0, tot = 0;
      for (int w = 0; w < kThreads / 32; ++w) {
        if (w < wid) wb += S.warp_cnt[w];
        tot += S.warp_cnt[w];
      }
      const uint32_t rank = running + wb + __popc(m & ((1u << lane) - 1));
      append_sel(f && rank < quota, (int32_t)i, nsel0, sel0, lane);
      running += tot;
      __syncthreads();
    }
  }
  cluster_sync();

  if (crank != 0) return;
  // CTA 0: map to positions, sort ascending, write (-1 padded)
  const uint32_t n = min(S.n_sel, (uint32_t)r.k);
  int32_t *out = r.out + (int64_t)row * r.k;
  for (uint32_t i = tid; i < n; i += kThreads) {
    const int32_t s = S.sel[i];
    int32_t pos = s;
    if (r.pool) {
      const int32_t blk = __ldg(r.pool + (int64_t)row * r.pool_stride + s / BLOCK);
      pos = blk * BLOCK + (s & (BLOCK - 1));
    }
    S.sel[i] = pos;
  }
  __syncthreads();
  for (uint32_t i = tid; i < n; i += kThreads) {
    const int32_t v = S.sel[i];
    uint32_t rank = 0;
    for (uint32_t j = 0; j < n; ++j) rank += S.sel[j] < v;
    out[rank] = v;
  }
  for (int i = (int)n + tid; i < r.k; i += kThreads) out[i] = -1;
}

}  // namespace

bool topk_cluster_supported(const TopkRows &r) { return r.k <= kSelMax; }

cudaError_t launch_topk_cluster(const TopkRows &r, cudaStream_t stream, int *launches) {
  if (r.rows <= 0) return cudaSuccess;
  static int max_cluster = 0;
  if (!max_cluster) {
    max_cluster = 8;
    if (cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
        cudaSuccess)
      max_cluster = 16;
    else
      (void)cudaGetLastError();
  }
  const size_t smem = sizeof(TopkClusterSmem) + 16;
  cudaError_t err = cudaFuncSetAttribute(topk_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  int64_t c = (r.row_len + 8191) / 8192;
  if (c < 1) c = 1;
  if (c > max_cluster) c = max_cluster;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)c, (unsigned)r.rows, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, topk_cluster_kernel, r);
  if (err == cudaSuccess) ++*launches;
  return err;
}

}  // namespace csa2
