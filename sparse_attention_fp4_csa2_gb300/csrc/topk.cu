// Batched exact top-K by radix select: the index_topk = 512 highest indexer
// scores of a sequence, and the candidate_topk_blocks = 2048 highest HSI block
// scores ("DeepSeek-V4.1-Flash - Architecture", sections 2 and 3;
// "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression", 2.3.4).
//
// Values become order-preserving 32-bit keys; ties are broken toward the lower
// index by selecting on the 64-bit composite (key << 32 | ~index), which is
// unique, so the result is deterministic.  -inf marks an invalid slot.
//
//   1. histogram   (many CTAs per row): 2048-bin histogram of the top 11 key
//      bits, warp-aggregated shared-memory counts flushed to global.
//   2. select      (many CTAs per row): every CTA finds the threshold bin T
//      from the row histogram; keys above T are selected outright (fewer than
//      K of them), keys in T are appended to a candidate list.
//   3. finish      (one CTA per row): radix select of the remaining count among
//      the candidates on the low 53 composite bits (8-bit digits, in shared
//      memory when they fit), then the K winners are mapped to positions
//      (through the HSI pool for Reindex rows), sorted ascending and written,
//      -1 padded.
// Rows are streamed once by passes 1 and 2 (4 B per position each, against
// the sweep's 256 B).  The HSI pool (k <= 2048) goes to the cluster top-K
// instead (launch_pool_topk); this path serves larger pools.
#include "kernels.cuh"

namespace csa2 {

namespace {

constexpr int kHistThreads = 256;
constexpr int kPerThread = 16;
constexpr int kChunk = kHistThreads * kPerThread;   // 4096 values per CTA
constexpr int kFinThreads = 1024;
constexpr int kCandSmem = 12288;                    // candidates kept in shared memory
constexpr int kRankMax = 2048;                      // rank-by-counting below this many

__device__ __forceinline__ uint32_t row_force_index(const TopkRows &r, int row) {
  if (!r.force_nvis) return 0xFFFFFFFFu;
  int32_t nv = __ldg(r.force_nvis + row);
  if (nv > r.n_max) nv = (int32_t)r.n_max;
  if (nv <= 0) return 0xFFFFFFFFu;
  return (uint32_t)((nv - 1) / r.force_block);
}

// All kPerThread keys of this thread's share of a chunk, loads issued together.
__device__ __forceinline__ void load_keys(const TopkRows &r, const float *row, int64_t c0, uint32_t force,
                                          uint32_t (&keys)[kPerThread]) {
  float v[kPerThread];
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int64_t i = c0 + j * kHistThreads + threadIdx.x;
    v[j] = (i < r.row_len) ? row[i] : -INFINITY;
  }
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int64_t i = c0 + j * kHistThreads + threadIdx.x;
    keys[j] = ((uint32_t)i == force && i < r.row_len) ? f32_key(INFINITY)
              : (v[j] == -INFINITY || v[j] != v[j]) ? 0u : f32_key(v[j]);
  }
}

__global__ void __launch_bounds__(kHistThreads) topk_hist_kernel(const TopkRows r, TopkScratch s) {
  __shared__ uint32_t hist[TOPK_BINS];
  pdl_wait();   // the inputs' producer is complete past here (programmatic launch)
  const int row = blockIdx.y;
  for (int i = threadIdx.x; i < TOPK_BINS; i += kHistThreads) hist[i] = 0;
  __syncthreads();
  const float *vals = r.vals + (int64_t)row * r.row_stride;
  const uint32_t force = row_force_index(r, row);
  const int64_t c0 = (int64_t)blockIdx.x * kChunk;
  const int lane = threadIdx.x & 31;
  uint32_t keys[kPerThread];
  load_keys(r, vals, c0, force, keys);
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const uint32_t bin = keys[j] ? (keys[j] >> 21) : (uint32_t)TOPK_BINS;  // sentinel: nothing to count
    const uint32_t peers = __match_any_sync(0xffffffffu, bin);
    if (bin < TOPK_BINS && lane == __ffs(peers) - 1) atomicAdd(&hist[bin], (uint32_t)__popc(peers));
  }
  __syncthreads();
  uint32_t *gh = s.hist + (int64_t)row * TOPK_BINS;
  for (int i = threadIdx.x; i < TOPK_BINS; i += kHistThreads)
    if (hist[i]) atomicAdd(gh + i, hist[i]);
}

// Threshold bin of a row from its histogram: the bin T holding the k-th
// largest key, with above = number of keys in bins > T.  T = -1 when the row
// has at most k valid keys (everything is selected).
__device__ void find_threshold(const uint32_t *gh, int k, int *T_out, uint32_t *above_out, uint32_t *smem_scan) {
  // thread t owns the 8 bins [2047 - 8t, 2040 - 8t] (descending), 256 threads
  const int t = threadIdx.x;
  uint32_t c[8], local = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    c[j] = gh[TOPK_BINS - 1 - (8 * t + j)];
    local += c[j];
  }
  // exclusive scan of `local` over threads in order t = 0..255
  const int lane = t & 31, wid = t >> 5;
  uint32_t incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) smem_scan[wid] = incl;
  __syncthreads();
  uint32_t wbase = 0, total = 0;
  for (int w = 0; w < kHistThreads / 32; ++w) {
    if (w < wid) wbase += smem_scan[w];
    total += smem_scan[w];
  }
  uint32_t before = wbase + incl - local;
  if (t == 0) {
    *T_out = -1;
    *above_out = total;
  }
  __syncthreads();
  if (total > (uint32_t)k) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (before < (uint32_t)k && before + c[j] >= (uint32_t)k) {
        *T_out = TOPK_BINS - 1 - (8 * t + j);
        *above_out = before;
      }
      before += c[j];
    }
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kHistThreads) topk_select_kernel(const TopkRows r, TopkScratch s) {
  __shared__ uint32_t scan[kHistThreads / 32];
  __shared__ int T_sh;
  __shared__ uint32_t above_sh;
  pdl_wait();   // the histograms are complete past here (programmatic launch)
  const int row = blockIdx.y;
  find_threshold(s.hist + (int64_t)row * TOPK_BINS, r.k, &T_sh, &above_sh, scan);
  const int T = T_sh;
  uint32_t *cnt = s.counters + (int64_t)row * 4;
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    cnt[2] = (uint32_t)(T + 1);
    cnt[3] = above_sh;
  }
  const float *vals = r.vals + (int64_t)row * r.row_stride;
  const uint32_t force = row_force_index(r, row);
  int32_t *sel = s.sel + (int64_t)row * r.k;
  uint64_t *cand = s.cand + (int64_t)row * r.row_len;
  const int64_t c0 = (int64_t)blockIdx.x * kChunk;
  const int lane = threadIdx.x & 31;
  uint32_t keys[kPerThread];
  load_keys(r, vals, c0, force, keys);
#pragma unroll
  for (int j = 0; j < kPerThread; ++j) {
    const int64_t i = c0 + j * kHistThreads + threadIdx.x;
    const uint32_t key = keys[j];
    const int bin = key ? (int)(key >> 21) : -2;
    const bool take = key && bin > T;
    const bool maybe = key && bin == T;
    const uint32_t mt = __ballot_sync(0xffffffffu, take);
    const uint32_t mm = __ballot_sync(0xffffffffu, maybe);
    uint32_t bt = 0, bm = 0;
    if (lane == 0) {
      if (mt) bt = atomicAdd(cnt + 0, (uint32_t)__popc(mt));
      if (mm) bm = atomicAdd(cnt + 1, (uint32_t)__popc(mm));
    }
    bt = __shfl_sync(0xffffffffu, bt, 0);
    bm = __shfl_sync(0xffffffffu, bm, 0);
    const uint32_t below = (1u << lane) - 1;
    if (take) {
      const uint32_t p = bt + __popc(mt & below);
      if (p < (uint32_t)r.k) sel[p] = (int32_t)i;
    }
    if (maybe) {
      const uint32_t p = bm + __popc(mm & below);
      cand[p] = ((uint64_t)key << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)i);
    }
  }
}

__device__ __forceinline__ int32_t map_out(const TopkRows &r, int row, int32_t i) {
  if (!r.pool) return i;
  const int32_t blk = __ldg(r.pool + (int64_t)row * r.pool_stride + i / BLOCK);
  return blk * BLOCK + (i & (BLOCK - 1));
}

__global__ void __launch_bounds__(kFinThreads) topk_finish_kernel(const TopkRows r, TopkScratch s) {
  extern __shared__ uint64_t fin_smem[];
  uint64_t *cs = fin_smem;                                      // [kCandSmem]
  int32_t *list = reinterpret_cast<int32_t *>(cs + kCandSmem);  // [pow2 >= k]
  __shared__ uint32_t hist[256];
  __shared__ uint32_t n_list;
  __shared__ int digit_sh;
  __shared__ uint32_t above_sh;
  __shared__ int last_sh;
  pdl_wait();   // the selection counts are complete past here (programmatic launch)

  const int row = blockIdx.x;
  const uint32_t *cnt = s.counters + (int64_t)row * 4;
  const uint32_t n_sel = min(cnt[0], (uint32_t)r.k);
  const uint32_t n_cand = cnt[1];
  const int T = (int)cnt[2] - 1;
  const uint32_t above = cnt[3];
  const int32_t *sel = s.sel + (int64_t)row * r.k;
  const uint64_t *gc = s.cand + (int64_t)row * r.row_len;

  int P = 1;
  while (P < r.k) P <<= 1;
  for (int i = threadIdx.x; i < P; i += kFinThreads) list[i] = (i < (int)n_sel) ? sel[i] : 0x7FFFFFFF;
  if (threadIdx.x == 0) n_list = n_sel;
  uint32_t need = (T >= 0) ? (uint32_t)r.k - min(above, (uint32_t)r.k) : 0u;
  const bool in_smem = n_cand <= (uint32_t)kCandSmem;
  if (in_smem)
    for (uint32_t i = threadIdx.x; i < n_cand; i += kFinThreads) cs[i] = gc[i];
  const uint64_t *c = in_smem ? cs : gc;
  __syncthreads();

  if (in_smem && n_cand <= (uint32_t)kRankMax && need > 0) {
    // few candidates: rank each by counting larger composites (all distinct)
    for (uint32_t i = threadIdx.x; i < n_cand; i += kFinThreads) {
      const uint64_t v = c[i];
      uint32_t rank = 0;
      for (uint32_t j = 0; j < n_cand; ++j) rank += c[j] > v;
      if (rank < need) list[n_sel + rank] = (int32_t)(0xFFFFFFFFu - (uint32_t)(v & 0xFFFFFFFFull));
    }
    if (threadIdx.x == 0) n_list = n_sel + min(need, n_cand);
    need = 0;
  }
  // radix select of `need` largest among the candidates on bits 55..0
  // (the top 11 key bits are equal for all of them)
  uint64_t prefix = 0;
  for (int shift = 48; shift >= 0 && need > 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kFinThreads) hist[i] = 0;
    __syncthreads();
    for (uint32_t i = threadIdx.x; i < n_cand; i += kFinThreads) {
      const uint64_t v = c[i] & 0x00FFFFFFFFFFFFFFull;
      if ((v >> (shift + 8)) == prefix) atomicAdd(&hist[(v >> shift) & 255], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // descending scan over 256 digits by one warp: lane l owns digits 255-8l .. 248-8l
      const int lane = threadIdx.x;
      uint32_t h[8], loc = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        h[j] = hist[255 - (8 * lane + j)];
        loc += h[j];
      }
      uint32_t incl = loc;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      uint32_t before = incl - loc;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (before < need && before + h[j] >= need) {
          digit_sh = 255 - (8 * lane + j);
          above_sh = before;
          last_sh = (before + h[j] == need) ? 1 : 0;
        }
        before += h[j];
      }
    }
    __syncthreads();
    const int d = digit_sh;
    const uint32_t ab = above_sh;
    const int last = last_sh;   // the whole digit-d bucket is needed: finish here
    // emit every candidate of this prefix with a larger digit (or >= d when last)
    for (uint32_t i = threadIdx.x; i < n_cand; i += kFinThreads) {
      const uint64_t v = c[i] & 0x00FFFFFFFFFFFFFFull;
      if ((v >> (shift + 8)) == prefix && (int)((v >> shift) & 255) >= d + 1 - last) {
        const uint32_t p = atomicAdd(&n_list, 1u);
        if (p < (uint32_t)r.k) list[p] = (int32_t)(0xFFFFFFFFu - (uint32_t)(c[i] & 0xFFFFFFFFull));
      }
    }
    need = last ? 0u : need - ab;
    prefix = (prefix << 8) | (uint64_t)d;
    if (shift == 0 && need > 0) {
      // the composite equal to the full prefix is unique
      if (threadIdx.x == 0) {
        const uint32_t p = atomicAdd(&n_list, 1u);
        if (p < (uint32_t)r.k) list[p] = (int32_t)(0xFFFFFFFFu - (uint32_t)(prefix & 0xFFFFFFFFull));
      }
      need = 0;
    }
    __syncthreads();
  }
  __syncthreads();
  // map to output positions, then sort ascending (padding = INT_MAX)
  const uint32_t n_final = min(n_list, (uint32_t)r.k);
  int32_t *out = r.out + (int64_t)row * r.k;
  if (n_final <= (uint32_t)kRankMax) {
    // rank sort: distinct positions, each placed by counting the smaller ones
    int32_t mine[kRankMax / kFinThreads];
    int cnt = 0;
    for (uint32_t i = threadIdx.x; i < n_final; i += kFinThreads) mine[cnt++] = map_out(r, row, list[i]);
    __syncthreads();
    cnt = 0;
    for (uint32_t i = threadIdx.x; i < n_final; i += kFinThreads) list[i] = mine[cnt++];
    __syncthreads();
    cnt = 0;
    for (uint32_t i = threadIdx.x; i < n_final; i += kFinThreads) {
      const int32_t v = list[i];
      uint32_t rank = 0;
      for (uint32_t j = 0; j < n_final; ++j) rank += list[j] < v;
      out[rank] = v;
    }
    for (int i = (int)n_final + threadIdx.x; i < r.k; i += kFinThreads) out[i] = -1;
    return;
  }
  for (int i = threadIdx.x; i < P; i += kFinThreads)
    list[i] = (i < (int)n_final) ? map_out(r, row, list[i]) : 0x7FFFFFFF;
  __syncthreads();
  for (int k2 = 2; k2 <= P; k2 <<= 1) {
    for (int j = k2 >> 1; j > 0; j >>= 1) {
      for (int i = threadIdx.x; i < P; i += kFinThreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const int32_t a = list[i], b = list[ixj];
          const bool up = (i & k2) == 0;
          if ((a > b) == up) {
            list[i] = b;
            list[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int i = threadIdx.x; i < r.k; i += kFinThreads) out[i] = (i < (int)n_final) ? list[i] : -1;
}

// Rows of block scores with the forced block set to +inf, padded with -inf
// to `stride` (a multiple of 4) values: the input of the cluster top-K.
__global__ void __launch_bounds__(256) pool_force_copy_kernel(const TopkRows r, float *dst, int64_t stride) {
  pdl_wait();   // the block scores' producer is complete past here (programmatic launch)
  const int row = blockIdx.y;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= stride) return;
  const uint32_t force = row_force_index(r, row);
  float v = -INFINITY;
  if (i < r.row_len) v = (uint32_t)i == force ? INFINITY : __ldg(r.vals + (int64_t)row * r.row_stride + i);
  dst[(int64_t)row * stride + i] = v;
}

}  // namespace

cudaError_t launch_pool_topk(const TopkRows &r, void *scratch, int num_sms, cudaStream_t stream, int *launches) {
  if (r.rows <= 0) return cudaSuccess;
  if (r.k > 2048) return launch_topk(r, carve_topk_scratch(scratch, r.rows, r.row_len, r.k), num_sms, stream, launches);
  // the cluster top-K over a forced copy (rows x stride floats fit in the
  // scratch: topk_scratch_bytes holds 8 B per value plus 8 KB per row)
  const int64_t stride = (r.row_len + 3) & ~int64_t(3);
  float *copy = static_cast<float *>(scratch);
  if (stride > 0) {
    dim3 grid((unsigned)((stride + 255) / 256), (unsigned)r.rows);
    cudaError_t err = launch_pdl(pool_force_copy_kernel, grid, dim3(256), 0, stream, 0u, r, copy, stride);
    if (err != cudaSuccess) return err;
    ++*launches;
  }
  TopkRows c = r;
  c.vals = copy;
  c.row_len = stride;
  c.row_stride = stride;
  c.force_nvis = nullptr;
  return launch_topk(c, stream, launches, /*profiled*/ false);
}

size_t topk_scratch_bytes(int32_t rows, int64_t row_len, int32_t k) {
  size_t b = 0;
  b += (size_t)rows * TOPK_BINS * 4;
  b += (size_t)rows * 4 * 4;
  b = (b + 255) & ~size_t(255);
  b += (size_t)rows * k * 4;
  b = (b + 255) & ~size_t(255);
  b += (size_t)rows * row_len * 8;
  return (b + 255) & ~size_t(255);
}

TopkScratch carve_topk_scratch(void *base, int32_t rows, int64_t row_len, int32_t k) {
  uint8_t *p = static_cast<uint8_t *>(base);
  TopkScratch s;
  s.hist = reinterpret_cast<uint32_t *>(p);
  s.counters = s.hist + (size_t)rows * TOPK_BINS;
  size_t off = ((size_t)rows * TOPK_BINS * 4 + (size_t)rows * 16 + 255) & ~size_t(255);
  s.sel = reinterpret_cast<int32_t *>(p + off);
  off = (off + (size_t)rows * k * 4 + 255) & ~size_t(255);
  s.cand = reinterpret_cast<uint64_t *>(p + off);
  return s;
}

cudaError_t launch_topk(const TopkRows &r, const TopkScratch &s, int num_sms, cudaStream_t stream, int *launches) {
  (void)num_sms;
  if (r.rows <= 0) return cudaSuccess;
  cudaError_t err = cudaMemsetAsync(s.hist, 0, (size_t)r.rows * (TOPK_BINS * 4 + 16), stream);
  if (err != cudaSuccess) return err;
  const int64_t chunks = (r.row_len + kChunk - 1) / kChunk;
  if (chunks > 0) {
    dim3 grid((unsigned)chunks, (unsigned)r.rows);
    err = launch_pdl(topk_hist_kernel, grid, dim3(kHistThreads), 0, stream, 0u, r, s);
    if (err != cudaSuccess) return err;
    err = launch_pdl(topk_select_kernel, grid, dim3(kHistThreads), 0, stream, 0u, r, s);
    if (err != cudaSuccess) return err;
    *launches += 2;
  }
  int P = 1;
  while (P < r.k) P <<= 1;
  const size_t smem = (size_t)kCandSmem * 8 + (size_t)P * 4;
  err = cudaFuncSetAttribute(topk_finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  err = launch_pdl(topk_finish_kernel, dim3((unsigned)r.rows), dim3(kFinThreads), smem, stream, 0u, r, s);
  if (err != cudaSuccess) return err;
  ++*launches;
  return cudaSuccess;
}

}  // namespace csa2
