// Sparse-attention readout over gathered FP4 main-KV entries and the FP8 SWA
// window, on the 5th-generation tensor cores.
//
// For one query token: one softmax over {top-K main-KV entries} U {SWA rows},
// logits q_h . k_j / sqrt(512), key = value = the dequantised 512-d latent
// ("DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression", sections
// 3.3.1-3.3.2: key = value = content, a convex combination of the selected
// entries; "DeepSeek-V4.1-Flash - Architecture", section 2: 64 heads x 512,
// top-512 + SWA-128).  FP4 stores the cache; the values are dequantised before
// the products (section 2.4.4: FP4 reduces storage, not matmul cost).  E2M1 x
// E4M3 is exact in fp16, so the tensor cores see the dequantised values.
//
// Work split.  An item is one token's keys, or -- when the tokens are too few
// to fill the SMs -- one of C <= 8 chunks of them (a chunk takes an equal
// share of the top-K list and of the SWA rows).  With C = 1 the CTAs are
// persistent and walk the items; with C > 1 the C chunks of a token are the
// CTAs of one thread-block cluster: each loads a share of the token's Q for
// all of them (TMA multicast), and they merge their partial results through
// distributed shared memory.
//
// Inside a CTA an item's keys go through in blocks of up to 128 (a single
// block of up to 160 when every CTA holds one item).  Per block:
//   dequant   8 worker warps load the block's rows (FP4 entries through the
//             index list, or E4M3 SWA rows) into registers one block ahead,
//             then write them as fp16 into a 128B-swizzled K-major tile
//             [8 columns of 64 dims][rows][128 B], one column pair at a time;
//   S = Q K^T one thread of the MMA warp issues M = 64 (heads) x N = rows x
//             K = 512 as the column pairs land (S in TMEM, heads on lanes);
//   softmax   the workers read S per head (thread = head, two warps per head
//             split the keys), keep a running reference max per head that is
//             raised only when a block exceeds it by 2^8 (then O^T is rescaled
//             in TMEM), and write P (fp16, times the SWA row scale) K-major as
//             [64 heads][rows];
//   O^T      += V^T P^T: M = 128 dims (four blocks) x N = 64 heads x K = rows,
//             V^T read MN-major from the same tile; each 128-dim block's
//             commit frees its column pair for the next block's dequant.
// The MMA issue sequences are runtime loops with descriptors advanced by
// constants (small code: a CTA runs it once, with a cold instruction
// cache).  At an item's end the workers normalise O^T and write the output
// (C = 1) or the partial (C > 1) while the next item's first block is
// already multiplying.
//
// Every wait is bounded.  After a wait runs out the kernel records
// CSA2_DEV_ERR_TIMEOUT and falls through every later wait, so that all
// threads still meet at the same named and cluster barriers and the CTA
// exits; its output is then undefined.
// This unit is compiled without relocatable device code, so that ptxas
// allots each warp role the registers its setmaxnreg asks for (with
// separate compilation it ignores setmaxnreg); it keeps its own error word.
#define CSA2_WHOLE_PROGRAM_TU 1
#include "kernels.cuh"

namespace csa2 {

namespace {

constexpr int kWorkers = 256;                    // 8 worker warps (warpgroups 0 and 1)
constexpr int kThreads = kWorkers + 128;         // + warpgroup 2: the MMA warp and 3 idle warps
constexpr int kMmaWarp = kWorkers / 32;
// Register split (setmaxnreg): launched at 65536 / 384 -> 168 per thread; the
// MMA warpgroup gives up to 136, the workers take 184 (256 x 184 + 128 x 136
// = 64,512 = 384 x 168; per scheduler 2 x 184 + 136 = 504 <= 512).  Both
// roles then compile without spills.
constexpr uint32_t kRegsMma = 136, kRegsWork = 184;
constexpr int kQThreads = 96;                    // warps 9-11: convert each item's Q
static_assert(kWorkers * kRegsWork + 128 * kRegsMma <= kThreads * 168, "register split exceeds the launch budget");
constexpr int kMaxBk = 160;                      // rows of a single-block item
constexpr int kBlockRows = 128;                  // rows of a block of a multi-block item
constexpr int kTileRegion = kMaxBk * D * 2;      // 160 KB
constexpr int kQBytes = H * D * 2;               // 64 KB fp16 Q
constexpr int kAtom = H * 128;                   // 8 KB: a 64-row atom column (Q, P^T)
constexpr int kPOffMulti = kBlockRows * D * 2;   // P^T of multi-block items: in the tile region's tail
constexpr int kRedOffMulti = kPOffMulti + 3 * kAtom;
constexpr int kRedOffSingle = 3 * kAtom;         // single-block items: P^T and reductions in the Q region
// cluster combine, in the tile region: received [8][2][64] max / sum and
// [C][D / C rows][128 B] partials, [8][64] weights, staged rows to send
constexpr uint32_t kCombineParts = 8 * 2 * H * 4;
constexpr uint32_t kCombineWgt = kCombineParts + D * 128;
constexpr uint32_t kCombineStage = kCombineWgt + 8 * H * 4;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColO = 256;                  // O^T: columns 256 + 64 mt + head, lanes = dims
constexpr float kLazy = 8.0f;                    // log2 margin before the reference max is raised
constexpr float kLogit = 0.06375871295460785f;   // log2(e) / sqrt(512)
constexpr float kLn2 = 0.69314718055994531f;
constexpr uint32_t kIdescPV = idesc_f16(/*fp16*/ 0, /*A MN-major*/ 1, /*B K-major*/ 0, /*N*/ H, /*M*/ 128);

struct __align__(16) Ctl {
  uint64_t q_full[4], q_ready[4], s_full, p_full, done, comb;
  uint64_t cols_full[4], cols_free[4];
  uint32_t tmem_base;
  volatile uint32_t abort;
  __align__(16) float rs[kMaxBk];      // per row: 1 (main entry) or the SWA row scale
  __align__(16) uint8_t vld[kMaxBk];   // per row: holds a key
  float fac[H];            // O^T rescale factor per head (block being processed)
  float inv_l[H];          // per head at an item's end: 1 / row sum (0 if empty)
  float mfin[H];           // per head at an item's end: reference max (log2 units)
  float lfin[H];           // per head at an item's end: row sum
};

constexpr size_t kSmemBytes = 1024 + (size_t)kTileRegion + kQBytes + sizeof(Ctl);
static_assert(kSmemBytes <= 232448, "attention exceeds the shared-memory limit");
static_assert(kRedOffMulti + 2 * H * 4 <= kTileRegion, "multi-block reductions overflow the tile region");
static_assert(kCombineStage + D * 128 <= kTileRegion, "cluster combine overflows the tile region");
static_assert(kRedOffSingle >= (kMaxBk / 64 + 1) * kAtom && kRedOffSingle + 4 * H * 4 <= kQBytes,
              "single-block P^T overlaps the reductions");

// One item: a token and its chunk of keys.  Item key e < nW is SWA row
// w0 + e of the token's window; e >= nW is top-K slot k0 + e - nW.  (SWA rows
// first: in a block of more than 128 rows the rows past 128 are then entries.)
struct Item {
  int64_t gp;          // token (global problem index)
  int64_t seq_row0;    // first main-KV row of the token's sequence
  int64_t swa_row0;    // first SWA row of the token's window
  int swa_len;         // valid rows of the window
  int k0, nW, w0, R, nb;
};

__device__ __forceinline__ Item item_info(const AttnArgs &a, int item) {
  Item it;
  const int C = a.C;
  const int tok = item / C, c = item - tok * C;
  it.gp = a.p0 + tok;
  it.seq_row0 = (it.gp / a.tokens) * a.cap;
  it.k0 = (c * a.K) / C;
  it.w0 = (c * a.W) / C;
  it.nW = ((c + 1) * a.W) / C - it.w0;
  it.R = it.nW + ((c + 1) * a.K) / C - it.k0;
  it.nb = it.R > a.Bk ? (it.R + a.Bk - 1) / a.Bk : 1;
  if (a.causal_swa) {
    const int64_t seq = it.gp / a.tokens;
    const int64_t pos = a.first_pos + it.gp % a.tokens;
    const int64_t start = pos - a.W + 1 > 0 ? pos - a.W + 1 : 0;
    it.swa_row0 = seq * a.swa_seq_rows + (start - a.swa_first_pos);
    it.swa_len = (int)(pos - start + 1);
  } else {
    it.swa_row0 = it.gp * a.W;
    it.swa_len = a.W > 0 ? min(__ldg(a.swa_len + it.gp), a.W) : 0;
  }
  return it;
}

// Blocks of an item (its key count over the block size, at least one).
__device__ __forceinline__ int item_blocks(const AttnArgs &a, int item) {
  const int c = item % a.C;
  const int R = ((c + 1) * a.W) / a.C - (c * a.W) / a.C + ((c + 1) * a.K) / a.C - (c * a.K) / a.C;
  return R > a.Bk ? (R + a.Bk - 1) / a.Bk : 1;
}

// A row's data, loaded one block ahead.  FP4 entry: v[2p], v[2p+1] are the
// codes of column cp + 2p (32 bytes), v[8].{x,y,z,w} the scale words of the
// four columns.  SWA row: v[4p .. 4p+3] are the 64 E4M3 bytes of column cp + 2p.
// (dequant_front consumes the columns in order, shifting the rest forward.)
template <int N>
struct RowBufN {
  uint4 v[N];
  float scale;
  int kind;   // 0 none, 1 FP4 entry, 2 SWA row
};
using RowBuf = RowBufN<16>;    // an entry or a SWA row

// Top-K slot of item key e, or -1 (also for SWA rows).
__device__ __forceinline__ int32_t row_slot(const AttnArgs &a, const Item &it, int e) {
  if (e < it.nW || e >= it.R) return -1;
  return __ldg(a.idx + it.gp * a.K + it.k0 + (e - it.nW));
}

template <int N>
__device__ __forceinline__ void load_row(const AttnArgs &a, const Item &it, int e, int32_t id, int cp,
                                         RowBufN<N> &b) {
  b.kind = 0;
  b.scale = 0.0f;
  if (e >= it.R) return;
  if (e >= it.nW) {
    if (id < 0) return;
    if (id >= a.cap) {
      set_error(CSA2_DEV_ERR_INDEX);
      return;
    }
    const uint8_t *src = a.kv + (it.seq_row0 + id) * ENTRY_BYTES;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int c = cp + 2 * p;
      b.v[2 * p] = ld_nc_v4(src + 32 * c);
      b.v[2 * p + 1] = ld_nc_v4(src + 32 * c + 16);
    }
    const uint8_t *sp = src + 256 + 4 * cp;
    b.v[8] = make_uint4(ld_nc_u32(sp), ld_nc_u32(sp + 8), ld_nc_u32(sp + 16), ld_nc_u32(sp + 24));
    b.scale = 1.0f;
    b.kind = 1;
  } else if constexpr (N == 16) {
    const int t = it.w0 + e;
    if (t >= it.swa_len) return;
    const uint8_t *src = a.swa + (it.swa_row0 + t) * D;
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
      for (int u = 0; u < 4; ++u) b.v[4 * p + u] = ld_nc_v4(src + 64 * (cp + 2 * p) + 16 * u);
    b.scale = __uint_as_float(ld_nc_u32(a.swa_scale + it.swa_row0 + t));
    b.kind = 2;
  }
}

// The buffer's front column as fp16 into column c of row r of the tile
// (16-byte chunk i of the row's 128-byte segment at (i ^ (r & 7)) * 16);
// the buffer's next column then moves to the front.  (One instantiation
// walked four times: the kernel's code stays small enough for the
// instruction cache.)
template <int N>
__device__ __forceinline__ void dequant_front(uint8_t *tile, uint32_t col_stride, int r, int c, RowBufN<N> &b) {
  uint8_t *rowp = tile + (uint32_t)c * col_stride + (uint32_t)r * 128;
  const int sw = r & 7;
  if (b.kind == 1) {
    const uint32_t sc = b.v[8].x;
    const uint32_t w[8] = {b.v[0].x, b.v[0].y, b.v[0].z, b.v[0].w, b.v[1].x, b.v[1].y, b.v[1].z, b.v[1].w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      // 8 codes = 8 dims of scale group i / 2
      const uint32_t sb = (sc >> (8 * (i >> 1))) & 0xFFu;
      const uint32_t s2 = e4m3x2_to_half2((uint16_t)(sb | (sb << 8)));
      uint32_t h[4];
      e2m1x8_to_half2x4(w[i], h);
      const uint4 o = make_uint4(hmul2_u32(h[0], s2), hmul2_u32(h[1], s2), hmul2_u32(h[2], s2), hmul2_u32(h[3], s2));
      *reinterpret_cast<uint4 *>(rowp + ((i ^ sw) << 4)) = o;
    }
#pragma unroll
    for (int i = 0; i < 6; ++i) b.v[i] = b.v[i + 2];
    b.v[8] = make_uint4(b.v[8].y, b.v[8].z, b.v[8].w, 0u);
    return;
  }
  if constexpr (N == 16) {
    if (b.kind == 2) {
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 raw = b.v[u];
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        const uint4 o0 =
            make_uint4(e4m3x2_to_half2((uint16_t)(w[0] & 0xFFFF)), e4m3x2_to_half2((uint16_t)(w[0] >> 16)),
                       e4m3x2_to_half2((uint16_t)(w[1] & 0xFFFF)), e4m3x2_to_half2((uint16_t)(w[1] >> 16)));
        const uint4 o1 =
            make_uint4(e4m3x2_to_half2((uint16_t)(w[2] & 0xFFFF)), e4m3x2_to_half2((uint16_t)(w[2] >> 16)),
                       e4m3x2_to_half2((uint16_t)(w[3] & 0xFFFF)), e4m3x2_to_half2((uint16_t)(w[3] >> 16)));
        *reinterpret_cast<uint4 *>(rowp + (((2 * u) ^ sw) << 4)) = o0;
        *reinterpret_cast<uint4 *>(rowp + (((2 * u + 1) ^ sw) << 4)) = o1;
      }
#pragma unroll
      for (int i = 0; i < 12; ++i) b.v[i] = b.v[i + 4];
      return;
    }
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) *reinterpret_cast<uint4 *>(rowp + ((i ^ sw) << 4)) = make_uint4(0, 0, 0, 0);
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// Bounded wait that falls through once any role has given up.
__device__ __forceinline__ void wait_ft(Ctl &S, uint64_t *bar, uint32_t parity) {
  if (S.abort) return;
  if (!mbar_wait(bar, parity)) S.abort = 1;
}

// The next block a worker loads: with C = 1 the CTA strides through the
// items; with C > 1 it holds exactly one.
struct Cursor {
  int item, j;
  Item it;
  __device__ __forceinline__ void advance(const AttnArgs &a, int stride, int items) {
    if (++j >= it.nb) {
      j = 0;
      item += stride;
      if (item < items) it = item_info(a, item);
    }
  }
};

// The finished item's output: out = O^T / l (C = 1), or (C > 1) this chunk's
// (m, l) and its normalised partial (fp16, [dim][head]) for the dims the other
// chunks own; the merge follows a cluster barrier.
__device__ __forceinline__ void item_epilogue(const AttnArgs &a, Ctl &S, int item, uint32_t s_row, int tid, int q4,
                                              int wh, int lane) {
  const int64_t gp = a.p0 + item;   // C = 1: an item is a token
  bar_named(1, kWorkers);   // inv_l / mfin / lfin of the item are visible
  tc_fence_after();
  float *outp = a.out + gp * H * D;
#pragma unroll 1
  for (int mm = 0; mm < 2; ++mm) {
    const int mt = 2 * wh + mm;
    const int d = mt * 128 + 32 * q4 + lane;
    uint32_t v[2][32];
    tmem_ld32(s_row + kColO + (uint32_t)(mt * H), v[0]);
    tmem_ld32(s_row + kColO + (uint32_t)(mt * H + 32), v[1]);
    tmem_ld_wait();
    const float keep = S.abort ? 0.0f : 1.0f;
#pragma unroll
    for (int hh = 0; hh < H; ++hh) outp[hh * D + d] = __uint_as_float(v[hh >> 5][hh & 31]) * (S.inv_l[hh] * keep);
  }
  if (tid < H && a.lse)
    a.lse[gp * H + tid] = S.lfin[tid] > 0.0f ? (S.mfin[tid] + log2f(S.lfin[tid])) * kLn2 : -INFINITY;
}

// C > 1: the C chunks of a token are the CTAs of one cluster (rank = chunk),
// each the owner of D / C dims of the output.  Each CTA stages, in its own
// tile region, its row-normalised O for every other owner's dims (fp16,
// 128-byte rows [dim][64 heads], 16-byte chunks XOR-swizzled by the row) and
// its per-head reference max and row sum.  Once every CTA's products are done
// (a cluster barrier: the tile regions are free), thread c sends owner c its
// rows and the max / sum by bulk shared-to-shared copies that complete on the
// owner's `comb` barrier (the copies to the C - 1 owners go out in
// parallel).  Each owner then combines the C partials with the weights
// l_c 2^(m_c - M) / L -- one softmax over the union of the chunks' keys --
// and writes its dims; rank 0 also writes the log-sum-exp.  A second cluster
// barrier, arrived once a CTA has received everything and awaited at its
// end, keeps every CTA resident until the copies out of it are complete
// (residency only: its arrive orders nothing).
__device__ __forceinline__ void cluster_combine(const AttnArgs &a, Ctl &S, uint8_t *tile, uint32_t tmem, int item,
                                                int tid, int warp, int lane) {
  const int C = a.C;
  const int tok = item / C;
  const uint32_t rank = (uint32_t)(item - tok * C);
  const int64_t gp = a.p0 + tok;
  const int dc = D / C;                              // dims per owner (>= 64: a warp's 32 dims have one owner)
  const uint32_t slot = (uint32_t)dc * 128;          // one source's rows
  float(*mlr)[2][H] = reinterpret_cast<float(*)[2][H]>(tile);            // received: [source][max, sum][head]
  uint8_t *parts = tile + kCombineParts;                                  // received: [source][row][128 B]
  float(*wgt)[H] = reinterpret_cast<float(*)[H]>(tile + kCombineWgt);     // [source][head]
  uint8_t *stage = tile + kCombineStage;                                  // sent: [owner][row][128 B]
  const int q4 = warp & 3, wh = warp >> 2;
  const uint32_t s_row = tmem + ((uint32_t)(32 * q4) << 16);

  if (tid == 0) mbar_arrive_expect_tx(&S.comb, (uint32_t)(C - 1) * (slot + 2 * H * 4));
  if (tid < H) {
    mlr[rank][0][tid] = S.mfin[tid];   // sent to the peers from here, and this CTA's own
    mlr[rank][1][tid] = S.lfin[tid];
  }
  tc_fence_after();
#pragma unroll 1
  for (int mm = 0; mm < 2; ++mm) {
    const int mt = 2 * wh + mm;
    const int d = mt * 128 + 32 * q4 + lane;
    const int owner = d / dc;
    if (owner == (int)rank) continue;
    uint32_t v[2][32];
    tmem_ld32(s_row + kColO + (uint32_t)(mt * H), v[0]);
    tmem_ld32(s_row + kColO + (uint32_t)(mt * H + 32), v[1]);
    tmem_ld_wait();
    const int row = d - owner * dc;
    uint8_t *dst = stage + owner * slot + (uint32_t)row * 128;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t *w = &v[k >> 2][(k & 3) * 8];
      const float *il = S.inv_l + 8 * k;
      *reinterpret_cast<uint4 *>(dst + ((k ^ (row & 7)) << 4)) =
          make_uint4(pack_half2(__uint_as_float(w[0]) * il[0], __uint_as_float(w[1]) * il[1]),
                     pack_half2(__uint_as_float(w[2]) * il[2], __uint_as_float(w[3]) * il[3]),
                     pack_half2(__uint_as_float(w[4]) * il[4], __uint_as_float(w[5]) * il[5]),
                     pack_half2(__uint_as_float(w[6]) * il[6], __uint_as_float(w[7]) * il[7]));
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
  cluster_arrive();
  cluster_wait();   // every CTA's products are done and its rows staged
  if (tid < C && tid != (int)rank) {
    const uint32_t bar = dsmem_addr(&S.comb, (uint32_t)tid);
    bulk_s2s_cluster(dsmem_addr(parts + rank * slot, (uint32_t)tid), stage + tid * slot, slot, bar);
    bulk_s2s_cluster(dsmem_addr(&mlr[rank][0][0], (uint32_t)tid), &mlr[rank][0][0], 2 * H * 4, bar);
  }
  wait_ft(S, &S.comb, 0);   // every peer's rows and max / sum have landed
  __syncwarp();
  cluster_arrive_relaxed();   // (awaited at the end)
  if (tid < H) {
    float mc[8], lc[8];
    float M = -INFINITY;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      mc[c] = c < C ? mlr[c][0][tid] : -INFINITY;
      lc[c] = c < C ? mlr[c][1][tid] : 0.0f;
      M = fmaxf(M, mc[c]);
    }
    float L = 0.0f;
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      lc[c] = mc[c] == -INFINITY ? 0.0f : lc[c] * exp2f(mc[c] - M);
      L += lc[c];
    }
    const float invL = L > 0.0f ? 1.0f / L : 0.0f;
#pragma unroll
    for (int c = 0; c < 8; ++c)
      if (c < C) wgt[c][tid] = lc[c] * invL;
    if (rank == 0 && a.lse) a.lse[gp * H + tid] = L > 0.0f ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
  bar_named(1, kWorkers);
  // this CTA's dims d, heads 32 wh .. + 31
  float *outp = a.out + gp * H * D;
  const float keep = S.abort ? 0.0f : 1.0f;
#pragma unroll 1
  for (int mt = 0; mt < 4; ++mt) {
    const int d = mt * 128 + 32 * q4 + lane;
    if (d / dc != (int)rank) continue;
    uint32_t v[32];
    tmem_ld32(s_row + kColO + (uint32_t)(mt * H + wh * 32), v);
    tmem_ld_wait();
    float acc[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) acc[i] = __uint_as_float(v[i]) * S.inv_l[wh * 32 + i] * wgt[rank][wh * 32 + i];
    const int row = d - (int)rank * dc;
#pragma unroll 1
    for (int c = 0; c < C; ++c) {
      if (c == (int)rank) continue;
      const uint8_t *src = parts + c * slot + (uint32_t)row * 128;
      const float *wc = wgt[c] + wh * 32;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 q = *reinterpret_cast<const uint4 *>(src + (((4 * wh + k) ^ (row & 7)) << 4));
        const uint32_t q2[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&q2[e]));
          acc[8 * k + 2 * e] = fmaf(wc[8 * k + 2 * e], f.x, acc[8 * k + 2 * e]);
          acc[8 * k + 2 * e + 1] = fmaf(wc[8 * k + 2 * e + 1], f.y, acc[8 * k + 2 * e + 1]);
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 32; ++i) outp[(wh * 32 + i) * D + d] = acc[i] * keep;
  }
  __syncwarp();
  cluster_wait();
}

// Column pair p of an item's Q (16 KB: 64 heads x 128 dims): bf16 -> fp16 in
// place (the same 2-byte slots of the swizzled layout; |q| < 65504 assumed),
// once its copy has landed.
__device__ __forceinline__ void convert_q_pair(uint8_t *qs, int p, int t, int nthreads) {
  uint4 *q = reinterpret_cast<uint4 *>(qs + p * 2 * kAtom);
#pragma unroll 4
  for (int i = t; i < 2 * kAtom / 16; i += nthreads) {
    const uint4 v = q[i];
    q[i] = make_uint4(pack_half2(__uint_as_float(v.x << 16), __uint_as_float(v.x & 0xFFFF0000u)),
                      pack_half2(__uint_as_float(v.y << 16), __uint_as_float(v.y & 0xFFFF0000u)),
                      pack_half2(__uint_as_float(v.z << 16), __uint_as_float(v.z & 0xFFFF0000u)),
                      pack_half2(__uint_as_float(v.w << 16), __uint_as_float(v.w & 0xFFFF0000u)));
  }
  fence_proxy_async_smem();
}

// O^T (+)= V^T P^T for one block of nks x 16 keys over the four 128-dim
// blocks mt, in groups of G: within a group the key steps are the outer loop,
// so consecutive MMAs go to different accumulators (back-to-back MMAs into
// one accumulator wait for each other: 80-105 clocks per M128 N64 K16 MMA
// against 58-76 when four accumulators alternate).  Each group's commit frees
// its column pairs.  The key steps are a runtime loop with descriptors
// advanced by constants (no MMA sits under a per-instruction condition).
template <int G>
__device__ __forceinline__ void issue_pv(int nks, Ctl &S, uint32_t tmem, uint64_t vd, uint64_t pd, uint64_t cs16,
                                         uint32_t acc0) {
#pragma unroll 1
  for (int g0 = 0; g0 < 4; g0 += G) {
    uint64_t va = vd + 2 * g0 * cs16, pk = pd;
#pragma unroll 1
    for (int ks = 0; ks < nks; ++ks) {
      const uint32_t acc = (acc0 | (uint32_t)ks) ? 1u : 0u;
#pragma unroll
      for (int mt = 0; mt < G; ++mt)
        mma_f16(tmem + kColO + (uint32_t)((g0 + mt) * H), va + 2 * mt * cs16, pk, kIdescPV, acc);
      va += 128;   // 16 keys of the MN-major V^T
      pk += (ks & 3) == 3 ? (uint64_t)((kAtom >> 4) - 6) : 2ull;   // 16 keys of P^T; next atom after 64
    }
#pragma unroll
    for (int mt = 0; mt < G; ++mt) mma_commit(&S.cols_free[g0 + mt]);
  }
}

// Q of an item's token by TMA (bf16, 8 boxes of [64 heads x 64 dims], 128B swizzle).
__device__ __forceinline__ void load_q(const AttnArgs &a, Ctl &S, const CUtensorMap &tm_q, uint8_t *qs, int item) {
  const int64_t gp = a.p0 + item / a.C;
#pragma unroll
  for (int p = 0; p < 4; ++p) {   // one barrier per column pair: S starts on the first pair
    mbar_arrive_expect_tx(&S.q_full[p], (uint32_t)(2 * kAtom));
    tma_load_2d(qs + 2 * p * kAtom, &tm_q, 2 * p * 64, (int32_t)(gp * H), &S.q_full[p]);
    tma_load_2d(qs + (2 * p + 1) * kAtom, &tm_q, (2 * p + 1) * 64, (int32_t)(gp * H), &S.q_full[p]);
  }
}

// C > 1: the cluster's CTAs share one token, so CTA `rank` loads the column
// pairs p = rank (mod C) once for all of them (multicast); every CTA armed
// its four Q barriers before the cluster barrier that precedes this call.
__device__ __forceinline__ void load_q_cluster(const AttnArgs &a, Ctl &S, const CUtensorMap &tm_q, uint8_t *qs,
                                               int item) {
  const int tok = item / a.C;
  const int rank = item - tok * a.C;
  const int64_t gp = a.p0 + tok;
  const uint16_t mask = (uint16_t)((1u << a.C) - 1u);
#pragma unroll 1
  for (int p = rank; p < 4; p += a.C) {
    tma_load_2d_mc(qs + 2 * p * kAtom, &tm_q, 2 * p * 64, (int32_t)(gp * H), &S.q_full[p], mask);
    tma_load_2d_mc(qs + (2 * p + 1) * kAtom, &tm_q, (2 * p + 1) * 64, (int32_t)(gp * H), &S.q_full[p], mask);
  }
}

template <bool kSingle>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *tile = base;
  uint8_t *qs = base + kTileRegion;
  Ctl &S = *reinterpret_cast<Ctl *>(qs + kQBytes);
  // kSingle: every CTA holds one item of one block (up to 160 rows), and P^T
  // and the reductions live in the Q region once S has read Q
  uint8_t *pbuf = kSingle ? qs : tile + kPOffMulti;
  float(*red)[H] = reinterpret_cast<float(*)[H]>(kSingle ? qs + kRedOffSingle : tile + kRedOffMulti);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int items = a.problems * a.C;
  const int first_item = blockIdx.x;
  const int stride = gridDim.x;

  // The MMA warp's lane 0 sets up the barriers first.  C > 1: a cluster
  // barrier then orders every CTA's set-up before any Q multicast into it;
  // every thread arrives at once and awaits it once later (before its next
  // arrive).
  if (warp == kMmaWarp && lane == 0) {
    for (int p = 0; p < 4; ++p) {
      mbar_init(&S.q_full[p], 1);
      // one item per CTA (kSingle): the workers convert a share of Q too
      mbar_init(&S.q_ready[p], kSingle ? kWorkers + kQThreads : kQThreads);
    }
    mbar_init(&S.s_full, 1);
    mbar_init(&S.p_full, kWorkers);
    mbar_init(&S.done, 1);
    mbar_init(&S.comb, 1);
    for (int p = 0; p < 4; ++p) {
      // kSingle: warps 9 and 10 also write the rows past 128
      mbar_init(&S.cols_full[p], kSingle ? kWorkers + 64 : kWorkers);
      mbar_init(&S.cols_free[p], 1);
    }
    S.abort = 0;
    // C > 1: Q arrives by multicast from the cluster's CTAs (one item per CTA)
    if (a.C > 1)
      for (int p = 0; p < 4; ++p) mbar_arrive_expect_tx(&S.q_full[p], (uint32_t)(2 * kAtom));
    fence_barrier_init();
    prefetch_tmap(&tm_q);
  }
  __syncwarp();
  if (a.C > 1) cluster_arrive();
  // the previous kernel in the stream is complete past here (programmatic
  // launch: everything above touches only this CTA's shared memory)
  pdl_enter();

  // The first block's row of this thread: row tid / 2 for the workers, and
  // in a single block row 128 + (tid - 288) / 2 for warps 9 and 10
  // (entries: SWA rows come first).  Its top-K slot is requested first; the
  // MMA warp meanwhile sets up the barriers and TMEM and sends Q's loads.
  int e0 = -1;
  if (warp < kMmaWarp)
    e0 = tid >> 1;
  else if (kSingle && tid >= (kMmaWarp + 1) * 32 && tid < (kMmaWarp + 3) * 32)
    e0 = 128 + ((tid - (kMmaWarp + 1) * 32) >> 1);
  const bool row0 = first_item < items && e0 >= 0 && (warp < kMmaWarp || e0 < a.Bk);
  Item it0;
  int32_t id0 = -1;
  if (row0) {
    it0 = item_info(a, first_item);
    id0 = row_slot(a, it0, e0);
  }

  if (warp == kMmaWarp) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
    if (a.C > 1) cluster_wait();
    if (lane == 0 && first_item < items) {
      if (a.C > 1)
        load_q_cluster(a, S, tm_q, qs, first_item);
      else
        load_q(a, S, tm_q, qs, first_item);
    }
  }
  RowBuf b0;
  b0.kind = 0;
  b0.scale = 0.0f;
  if (row0) load_row(a, it0, e0, id0, tid & 1, b0);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  const uint32_t col_stride = (uint32_t)a.Bk * 128;   // bytes per 64-dim column of the tile
  // Each role sets its register budget at the head of its own branch (a
  // setmaxnreg before a join would bound the code after it by the lower one).
  if (warp >= kMmaWarp) {
   setmaxnreg_dec<kRegsMma>();
   if (warp > kMmaWarp) {
    // the other warps of the MMA warpgroup: every item's Q, bf16 -> fp16 in
    // place one column pair at a time as it lands (the MMA thread reloads Q
    // after an item's last S).  A single block (one item): Q lands before
    // the gathered rows, so the workers convert it with these warps first;
    // warps 9 and 10 then also write rows 128 .. (entries: SWA rows come
    // first).
    const int ht = tid - (kMmaWarp + 1) * 32;   // 0 .. 95
    if constexpr (kSingle) {
      const int r = 128 + (ht >> 1), hcp = ht & 1;
      const bool rows = ht < 64 && first_item < items && r < a.Bk;   // loaded into b0 at the start
      __syncwarp();
      if (a.C > 1) cluster_wait();
      if (first_item < items) {
#pragma unroll 1
        for (int p = 0; p < 4; ++p) {
          wait_ft(S, &S.q_full[p], 0);
          convert_q_pair(qs, p, kWorkers + ht, kWorkers + kQThreads);
          mbar_arrive(&S.q_ready[p]);
        }
        if (ht < 64) {
          if (rows && hcp == 0) {
            S.rs[r] = b0.scale;
            S.vld[r] = b0.kind != 0 ? 1 : 0;
          }
#pragma unroll 1
          for (int p = 0; p < 4; ++p) {
            if (rows) dequant_front(tile, col_stride, r, hcp + 2 * p, b0);
            fence_proxy_async_smem();
            mbar_arrive(&S.cols_full[p]);
          }
        }
      }
    } else {
      __syncwarp();
      if (a.C > 1) cluster_wait();
      uint32_t n = 0;
      for (int item = first_item; item < items; item += stride, ++n) {
#pragma unroll 1
        for (int p = 0; p < 4; ++p) {
          wait_ft(S, &S.q_full[p], n & 1u);
          convert_q_pair(qs, p, ht, kQThreads);
          mbar_arrive(&S.q_ready[p]);
        }
      }
    }
   } else {
    // ------------------------------------------------------------------ MMA
    if (lane == 0) {
      const uint32_t id_s = idesc_f16(/*fp16*/ 0, /*A K-major*/ 0, /*B K-major*/ 0, /*N*/ (uint32_t)a.Bk, /*M*/ 64);
      const uint64_t qd = smem_desc(smem_u32(qs), 16, 1024);
      const uint64_t td = smem_desc(smem_u32(tile), 16, 1024);
      const uint64_t vd = smem_desc(smem_u32(tile), col_stride, 1024);
      const uint64_t pd = smem_desc(smem_u32(pbuf), 16, 1024);
      const uint64_t cs16 = col_stride >> 4;
      const int nks = a.Bk / 16;
      uint32_t g = 0, n_item = 0;
      for (int item = first_item; item < items; item += stride, ++n_item) {
        const Item it = item_info(a, item);
        for (int j = 0; j < it.nb; ++j, ++g) {
          const uint32_t ph = g & 1u;

          // (no MMA sits under a per-instruction condition: a conditional
          // tcgen05.mma in unrolled code was observed to issue wrongly)
#pragma unroll 1
          for (int p = 0; p < 4; ++p) {
            if (j == 0) wait_ft(S, &S.q_ready[p], n_item & 1u);
            wait_ft(S, &S.cols_full[p], ph);
            tc_fence_after();
            const uint64_t a0 = qd + (uint64_t)(p * 2 * kAtom >> 4), a1 = a0 + (kAtom >> 4);
            const uint64_t b0 = td + 2 * p * cs16, b1 = b0 + cs16;
#pragma unroll
            for (int i = 0; i < 4; ++i) mma_f16(tmem, a0 + 2 * i, b0 + 2 * i, id_s, (p | i) ? 1u : 0u);
#pragma unroll
            for (int i = 0; i < 4; ++i) mma_f16(tmem, a1 + 2 * i, b1 + 2 * i, id_s, 1u);
          }
          mma_commit(&S.s_full);
          if (j == it.nb - 1 && item + stride < items) {
            // Q is read by the last block's S: reload it for the next item
            wait_ft(S, &S.s_full, ph);
            if (!S.abort) load_q(a, S, tm_q, qs, item + stride);
          }
          wait_ft(S, &S.p_full, ph);
          tc_fence_after();
          // single block: nothing waits for early column release; several
          // blocks: the next block's dequant starts on columns 0-3 early
          issue_pv<kSingle ? 4 : 2>(nks, S, tmem, vd, pd, cs16, j > 0 ? 1u : 0u);
        }
      }
      // every MMA of this CTA has completed before the teardown
      mma_commit(&S.done);
      wait_ft(S, &S.done, 0);
    }
   }
    if (a.C > 1) {   // the two cluster barriers of the combine
      cluster_arrive();
      cluster_wait();
      cluster_arrive();
      cluster_wait();
    }
  } else {
    setmaxnreg_inc<kRegsWork>();
    // -------------------------------------------------------------- workers
    const int cp = tid & 1;                          // columns cp, cp + 2, cp + 4, cp + 6
    const int r0 = tid >> 1;                         // row r0 of the block (rows past 128: warps 9, 10)
    const int q4 = warp & 3, wh = warp >> 2;         // TMEM lane quadrant, warp half
    const int th = lane >> 4;                        // thread half of the warp
    const int h = 16 * q4 + (lane & 15);             // head of this thread in the softmax
    const uint32_t s_row = tmem + ((uint32_t)(32 * q4) << 16);

    // the block being processed (item, block, blocks of the item); `ld`: the
    // next block to load into registers, whose top-K slot `ld_id` was
    // requested one block earlier
    int cur_item = first_item, cur_j = 0, cur_nb = 1;
    Cursor ld;
    ld.item = first_item;
    ld.j = 0;
    int32_t ld_id = -1;
    if (ld.item < items) {   // (the first block's row is in b0 already)
      ld.it = item_info(a, ld.item);
      cur_nb = ld.it.nb;
      if constexpr (!kSingle) {
        ld.advance(a, stride, items);
        if (ld.item < items) ld_id = row_slot(a, ld.it, ld.j * a.Bk + r0);
      }
    }
    __syncwarp();
    if (a.C > 1) cluster_wait();
    if constexpr (kSingle) {
      // Q (multicast or local TMA) lands before the gathered rows: this
      // thread's share of it first, while the rows are on their way
      if (first_item < items) {
#pragma unroll 1
        for (int p = 0; p < 4; ++p) {
          wait_ft(S, &S.q_full[p], 0);
          convert_q_pair(qs, p, tid, kWorkers + kQThreads);
          mbar_arrive(&S.q_ready[p]);
        }
      }
    }

    uint32_t g = 0, n_item = 0;
    bool epi_pending = false;
    int epi_item = 0;
    float m_ref = -INFINITY, l_part = 0.0f;

    for (; cur_item < items; ++g) {
      const uint32_t ph = g & 1u;
      const int j = cur_j;
      // ------------------------------------------------------ Q of a new item
      // --------------------------------------------------------- dequant
      if (cp == 0 && r0 < a.Bk) {
        S.rs[r0] = b0.scale;
        S.vld[r0] = b0.kind != 0 ? 1 : 0;
      }
#pragma unroll 1
      for (int p = 0; p < 4; ++p) {
        if (g > 0) wait_ft(S, &S.cols_free[p], (g - 1) & 1u);
        if (r0 < a.Bk) dequant_front(tile, col_stride, r0, cp + 2 * p, b0);
        fence_proxy_async_smem();
        mbar_arrive(&S.cols_full[p]);
      }
      // the finished item's epilogue overlaps this block's S = Q K^T
      if (epi_pending) {
        item_epilogue(a, S, epi_item, s_row, tid, q4, wh, lane);
        epi_pending = false;
      }
      // ------------------------------------------ next block into registers
      if constexpr (!kSingle) {
        if (ld.item < items) {
          load_row(a, ld.it, ld.j * a.Bk + r0, ld_id, cp, b0);
          ld.advance(a, stride, items);
          if (ld.item < items) ld_id = row_slot(a, ld.it, ld.j * a.Bk + r0);
        }
      }
      const int this_item = cur_item;
      const int this_nb = cur_nb;
      if (++cur_j >= cur_nb) {
        cur_j = 0;
        cur_item += stride;
        if (cur_item < items) cur_nb = item_blocks(a, cur_item);
      }
      // ---------------------------------------------------------- softmax
      // Thread (warp w, lane l) owns head h = 16 (w % 4) + l % 16 and the
      // 16-key slabs 2m + l / 16 of the slab pairs m = 2 mi + w / 4; one
      // 16x32bx2 load per pair brings both halves of the warp their slab.
      wait_ft(S, &S.s_full, ph);
      tc_fence_after();
      bar_named(1, kWorkers);   // rs / vld of every row are visible
      if (j == 0) {
        m_ref = -INFINITY;
        l_part = 0.0f;
      }
      constexpr int kPairs = kSingle ? 3 : 2;   // slab pairs per warp half (blocks of <= 160 / 128 rows)
      // Logits of slab pair mi for this thread: 16 keys from one 16x32bx2
      // load, the row scales and valid flags by 16-byte loads (no loads
      // under a condition: those serialise).  Slabs past the block read
      // neighbouring Ctl bytes, masked by k < Bk.  Two passes over TMEM (max,
      // then exponents) keep only one pair's values in registers.
      // The row scales and valid flags of slab pair mi's 16 keys, and the
      // logits from its TMEM values u.
      auto row_info = [&](int mi, float (&rsv)[16], uint32_t (&vb)[4]) {
        const int k0 = 16 * (2 * (2 * mi + wh) + th);
        const float4 *r4 = reinterpret_cast<const float4 *>(S.rs + k0);
        const uint4 v4 = *reinterpret_cast<const uint4 *>(S.vld + k0);
        vb[0] = v4.x;
        vb[1] = v4.y;
        vb[2] = v4.z;
        vb[3] = v4.w;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float4 f4 = r4[q];
          rsv[4 * q] = f4.x;
          rsv[4 * q + 1] = f4.y;
          rsv[4 * q + 2] = f4.z;
          rsv[4 * q + 3] = f4.w;
        }
      };
      auto apply = [&](int mi, const uint32_t (&u)[16], const float (&rsv)[16], const uint32_t (&vb)[4],
                       float (&x)[16]) {
        const int k0 = 16 * (2 * (2 * mi + wh) + th);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const bool ok = (k0 + i < a.Bk) && ((vb[i >> 2] >> (8 * (i & 3))) & 0xFFu);
          x[i] = ok ? __uint_as_float(u[i]) * (kLogit * rsv[i]) : -INFINITY;
        }
      };
      auto logits = [&](int mi, float (&x)[16]) {
        uint32_t u[16], vb[4];
        float rsv[16];
        tmem_ld16x2(s_row + (uint32_t)(32 * (2 * mi + wh)), u);
        row_info(mi, rsv, vb);   // overlaps the TMEM load
        tmem_ld_wait();
        apply(mi, u, rsv, vb, x);
      };
      // P = 2^(logit - m_ref) (x the SWA row scale) into P^T; the row sum
      // gathers the unscaled exponents.  `over` flags a logit above
      // m_ref + kLazy (the one-pass attempt below).
      auto store_p = [&](int mi, const float (&x)[16], float mref_s) {
        bool over = false;
        const int k0 = 16 * (2 * (2 * mi + wh) + th);
        uint32_t pk[8];
#pragma unroll
        for (int i = 0; i < 16; i += 2) {
          // masked keys hold -inf: 2^-inf = 0 (no branch); m_ref = -inf only when all are masked
          over |= (x[i] > mref_s + kLazy) | (x[i + 1] > mref_s + kLazy);
          const float p0 = ex2_approx(x[i] - mref_s), p1 = ex2_approx(x[i + 1] - mref_s);
          l_part += p0 + p1;
          const float2 r2 = *reinterpret_cast<const float2 *>(S.rs + k0 + i);
          pk[i >> 1] = pack_half2(p0 * r2.x, p1 * r2.y);
        }
        if (k0 < a.Bk) {
          // P^T K-major: [64-key atom column][64 heads][128 B]
          uint8_t *prow = pbuf + (k0 >> 6) * kAtom + h * 128;
          const int c0 = (k0 & 63) >> 3;
          *reinterpret_cast<uint4 *>(prow + ((c0 ^ (h & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
          *reinterpret_cast<uint4 *>(prow + (((c0 + 1) ^ (h & 7)) << 4)) = make_uint4(pk[4], pk[5], pk[6], pk[7]);
        }
        return over;
      };
      auto write_p = [&](float mref_s) {
        bool over = false;
#pragma unroll 1
        for (int mi = 0; mi < kPairs; ++mi) {
          float x[16];
          logits(mi, x);
          over |= store_p(mi, x, mref_s);
        }
        return over;
      };
      // After an item's first block the reference max is rarely raised: one
      // pass writes P with the current reference, and only if some logit is
      // above it by more than 2^kLazy (any thread) is the block redone by the
      // two passes below (max, then exponents).  Whether a reference exists
      // is the same for every head (it depends on which keys were valid).
      bool done_p = false;
      if constexpr (kSingle) {
        // one block (nothing accumulated yet): every logit of this thread
        // from one TMEM round trip, kept in registers for the max and the
        // exponents
        uint32_t u[kPairs][16];
#pragma unroll
        for (int mi = 0; mi < kPairs; ++mi) tmem_ld16x2(s_row + (uint32_t)(32 * (2 * mi + wh)), u[mi]);
        tmem_ld_wait();
        float x[kPairs][16];
        float mx = -INFINITY;
#pragma unroll
        for (int mi = 0; mi < kPairs; ++mi) {
          uint32_t vb[4];
          float rsv[16];
          row_info(mi, rsv, vb);
          apply(mi, u[mi], rsv, vb, x[mi]);
#pragma unroll
          for (int i = 0; i < 16; ++i) mx = fmaxf(mx, x[mi][i]);
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (th == 0) red[wh][h] = mx;
        bar_named(1, kWorkers);
        m_ref = fmaxf(red[0][h], red[1][h]);
        const float ms = m_ref == -INFINITY ? 0.0f : m_ref;
#pragma unroll
        for (int mi = 0; mi < kPairs; ++mi) (void)store_p(mi, x[mi], ms);
        done_p = true;
      } else {
        if (m_ref != -INFINITY) {
          const float l_save = l_part;
          const bool over = write_p(m_ref);
          done_p = !bar_named_or(2, kWorkers, over);
          if (!done_p) l_part = l_save;
        }
      }
      if (!done_p) {
        float mx = -INFINITY;
#pragma unroll 1
        for (int mi = 0; mi < kPairs; ++mi) {
          float x[16];
          logits(mi, x);
#pragma unroll
          for (int i = 0; i < 16; ++i) mx = fmaxf(mx, x[i]);
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
        if (th == 0) red[wh][h] = mx;
        bar_named(1, kWorkers);
        const float mc = fmaxf(red[0][h], red[1][h]);
        float f = 1.0f;
        if (m_ref == -INFINITY) {
          m_ref = mc;   // nothing accumulated yet
        } else if (mc > m_ref + kLazy) {
          f = exp2f(m_ref - mc);
          m_ref = mc;
        }
        if (th == 0 && wh == 0) S.fac[h] = f;
        const bool any = bar_named_or(2, kWorkers, f != 1.0f);
        if (any) {
          // O^T holds every earlier block (the dequant above waited for the
          // previous block's products): scale its head columns
          tc_fence_after();
#pragma unroll 1
          for (int mm = 0; mm < 2; ++mm) {
            const int mt = 2 * wh + mm;
#pragma unroll 1
            for (int hb = 0; hb < 2; ++hb) {
              uint32_t v[32];
              const uint32_t ta = s_row + kColO + (uint32_t)(mt * H + hb * 32);
              tmem_ld32(ta, v);
              tmem_ld_wait();
#pragma unroll
              for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * S.fac[hb * 32 + i]);
              tmem_st32(ta, v);
            }
          }
          tmem_st_wait();
        }
        l_part *= f;
        (void)write_p(m_ref == -INFINITY ? 0.0f : m_ref);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&S.p_full);

      if (j == this_nb - 1) {
        // ---------------------------------------------------- item finished
        // (kSingle: the sums take the next two rows, as no barrier separates
        // this from the reads of the maxima above)
        float(*red_l)[H] = red + (kSingle ? 2 : 0);
        const float lp = l_part + __shfl_xor_sync(0xffffffffu, l_part, 16);
        if (th == 0) red_l[wh][h] = lp;
        bar_named(1, kWorkers);
        if (th == 0 && wh == 0) {
          const float L = red_l[0][h] + red_l[1][h];
          S.lfin[h] = L;
          S.mfin[h] = m_ref;
          S.inv_l[h] = L > 0.0f ? 1.0f / L : 0.0f;
        }
        epi_pending = true;
        epi_item = this_item;
        ++n_item;
      }
    }
    if (epi_pending) {
      // the last item: wait for its products, then write (C = 1) or combine
      // across the cluster (C > 1: the CTA's one item)
      wait_ft(S, &S.cols_free[3], (g - 1) & 1u);
      if (a.C == 1) item_epilogue(a, S, epi_item, s_row, tid, q4, wh, lane);
    }
    if (a.C > 1) cluster_combine(a, S, tile, tmem, first_item, tid, warp, lane);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {   // the allocating warp
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

int device_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  return n;
}

// Clusters of `c` CTAs of the readout that can be resident at once (a
// cluster lives inside one GPC; one CTA per SM), from the occupancy query;
// the SM count over c when the query fails.  Cached per cluster size.
int max_active_clusters(int c, int sms) {
  static int cache[9] = {};
  if (c < 1 || c > 8) return 0;
  if (cache[c]) return cache[c];
  int n = 0;
  auto kern = sparse_attn_kernel<true>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)c, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)c;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes) != cudaSuccess ||
      cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    (void)cudaGetLastError();
    n = sms / c;
  }
  cache[c] = n;
  return n;
}

// Chunks per token: the most (1, 2, 4 or 8) whose clusters can all be
// resident at once (a second wave of clusters would double the launch),
// keeping at least 16 keys per chunk; 1 once the tokens fill the SMs.
// kernel 1 forces a split (C >= 2), kernel 2 a single chunk.
int choose_chunks(int problems, int K, int W, int kernel, int sms) {
  if (kernel == 2) return 1;
  int c = 1;
  for (int cand : {2, 4, 8})
    if ((int64_t)problems * cand <= sms && problems <= max_active_clusters(cand, sms) && (K + W) / cand >= 16)
      c = cand;
  if (kernel == 1 && c == 1) c = (K + W) >= 32 ? 2 : 1;
  return c;
}

}  // namespace

cudaError_t attn_take_error(unsigned int *bits) {
  unsigned int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_dev_error, sizeof(v));
  if (e == cudaSuccess && v) e = cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(zero));
  *bits = v;
  return e;
}

size_t attn_scratch_bytes(int32_t problems, int32_t K, int32_t W, int32_t kernel) {
  (void)problems;
  (void)K;
  (void)W;
  (void)kernel;
  return 256;   // the chunks of a token combine through distributed shared memory
}

cudaError_t launch_sparse_attn(AttnArgs a, void *scratch, cudaStream_t stream, int *launches) {
  if (a.problems <= 0) return cudaSuccess;
  const int sms = device_sms();
  a.C = choose_chunks(a.problems, a.K, a.W, a.kernel, sms);
  const int max_r = (a.K + a.C - 1) / a.C + (a.W + a.C - 1) / a.C;
  const int items = a.problems * a.C;
  const int grid = a.C > 1 ? items : (a.problems < sms ? a.problems : sms);
  const bool one_item = grid >= items;
  const int r16 = max_r > 16 ? (max_r + 15) / 16 * 16 : 16;
  // one block per CTA (its rows past 128 must be entries: SWA rows come first)
  const bool single = one_item && r16 <= kMaxBk && (a.W + a.C - 1) / a.C <= kBlockRows;
  a.Bk = single ? r16 : kBlockRows;
  (void)scratch;
  CUtensorMap tm_q;
  if (!make_tmap_bf16(&tm_q, a.q, D, (a.p0 + a.problems) * H, H)) return cudaErrorInvalidValue;
  auto kern = single ? sparse_attn_kernel<true> : sparse_attn_kernel<false>;
  cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  const ProfileEvents &pe = profile_events(CSA2_KERNEL_SPARSE_ATTN);
  if (pe.start && (err = record_profile_event(pe.start, stream)) != cudaSuccess) return err;
  err = launch_pdl(kern, dim3((unsigned)grid), dim3(kThreads), kSmemBytes, stream, (unsigned)a.C, tm_q, a);
  if (err != cudaSuccess) return err;
  ++*launches;
  if (pe.stop && (err = record_profile_event(pe.stop, stream)) != cudaSuccess) return err;
  return cudaSuccess;
}

}  // namespace csa2
