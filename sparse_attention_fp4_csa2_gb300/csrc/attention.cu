// Sparse-attention readout over gathered FP4 main-KV entries and the FP8 SWA
// window, on the 5th-generation tensor cores.
//
// For one query token: one softmax over {top-K main-KV entries} U {SWA rows},
// logits q_h . k_j / sqrt(512), key = value = the dequantised 512-d latent
// ("DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression", sections
// 3.3.1-3.3.2: key = value = content, a convex combination of the selected
// entries; "DeepSeek-V4.1-Flash - Architecture", section 2: 64 heads x 512,
// top-512 + SWA-128).  FP4 stores the cache; the values are dequantised before
// the products (section 2.4.4: FP4 reduces storage, not matmul cost).
//
// Work split (flash-decoding): a CTA owns 128 keys of one query token -- one
// chunk of the top-K list or of the SWA window -- and produces a partial (row
// max, row sum, output).  With up to 8 chunks (the pages' 512 + 128 keys make
// 5) the chunks of a token form one thread-block cluster and merge in shared
// memory: each CTA pushes to every other one, by bulk shared-to-shared copies,
// the slice of its normalised fp16 partial that CTA owns, and sums its own
// slice into the output; with more chunks the partials go to the workspace
// and a separate combine kernel merges them.  Inside a CTA:
//   gather   Q arrives by TMA and the SWA rows by one bulk copy (mbarrier);
//            every thread issues 16-byte cp.async copies of the selected FP4
//            entries (18 per 288-byte entry) into a shared staging area;
//   dequant  every thread turns its share of codes into fp16 (E2M1 x E4M3 is
//            exact in fp16) in a 128B-swizzled K-major tile [128 keys x 512];
//            SWA rows (E4M3) likewise from their staging area;
//   S^T      = K Q^T: 32 tcgen05 MMAs (M=128 keys, N=64 heads, K=16), fp32 in
//            TMEM; Q (bf16 -> fp16) sits in shared memory K-major;
//   softmax  each thread owns one key row of S^T for 32 heads; per-head max
//            and sum over the 128 keys by warp butterfly transposes + shared
//            memory; P = exp2(S - m) (times the SWA row scale) in fp16 written
//            MN-major [128 keys x 64 heads];
//   O        = P V: P as A (heads as M), the same shared tile read MN-major as
//            B (N = 2 x 256 dims, K = 128 keys); fp32 in TMEM with the heads
//            as lanes, so a thread reads 32 consecutive dims of one head;
//   merge    as above.
// Shared memory: 128 KB tile (the FP4 staging area lives in its tail and is
// consumed through registers before the tile is written; later the fp16
// partial), 64 KB Q (reused for P, then as the merge's receive area),
// reductions; one CTA per SM.  TMEM: 512 columns (S^T uses 128 of them, two
// accumulation chains, and is dead before O is written).
#include "kernels.cuh"

namespace csa2 {

namespace {

constexpr int kThreads = 256;
constexpr int kQBytes = H * D * 2;                  // 64 KB fp16
constexpr int kQAtomCol = H * 128;                  // 8 KB
constexpr int kMixSwa = 32;                         // SWA rows per chunk of the mixed layout
constexpr int kRedOff = 32768;                      // softmax reductions: in the Q region, past P

// Chunk layouts.  Split (kSwa = 0): a chunk is 128 top-K entries or 128 SWA
// rows.  Mixed (kSwa = 32): a chunk is 128 top-K entries and 32 SWA rows, so
// the pages' 512 + 128 keys make 4 chunks instead of 5 -- chosen when the
// chunks outnumber the SMs.  The tile is [8 columns of 64 dims][rows][128 B].
template <int kSwa>
struct Layout {
  static constexpr int kRows = ATTN_CHUNK + kSwa;
  static constexpr int kTileBytes = kRows * D * 2;                          // fp16 tile
  static constexpr int kAtomCol = kRows * 128;                             // one 64-dim column
  static constexpr int kStageOff = kTileBytes - ATTN_CHUNK * ENTRY_BYTES;  // FP4 staging at the tile's tail
  static constexpr int kSwaStageOff = kTileBytes - ATTN_CHUNK * D;         // split: SWA staging, upper half
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kIdescQK = idesc_f16(/*fp16*/ 0, /*A K-major*/ 0, /*B K-major*/ 0, /*N*/ H, /*M*/ ATTN_CHUNK);
// O = P V: A = P (M = 128 rows: the 64 heads, then 64 rows nobody reads), B = V
// read MN-major from the tile, N = 256 dims per instruction
constexpr uint32_t kPVN = 256;
constexpr uint32_t kIdescPV = idesc_f16(/*fp16*/ 0, /*A MN-major*/ 1, /*B MN-major*/ 1, /*N*/ kPVN, /*M*/ 128);

constexpr int kMaxClusterChunks = 8;   // portable cluster size
// cluster merge: the [64 heads x 512 dims] fp16 partial is 512 groups of 128 B
constexpr int kRowBytes = D * 2;
constexpr int kGroups = H * kRowBytes / 128;

struct __align__(16) AttnSmem {
  float mfin[H];   // mfin, lfin adjacent: one 512-byte (m, l) record per chunk
  float lfin[H];
  uint64_t bar_load;
  uint64_t bar_mma;
  uint64_t bar_ml;
  uint64_t bar_merge;
  uint32_t tmem_base;
  uint32_t vmask[(ATTN_CHUNK + kMixSwa) / 32];
  int32_t ids[ATTN_CHUNK];
  float row_scale[ATTN_CHUNK + kMixSwa];
};

// cluster merge scratch, in the tile region behind the 64 KB fp16 partial
struct MergeSmem {
  float ml_in[kMaxClusterChunks][2][H];   // every chunk's (m, l)
  float wgt[kMaxClusterChunks][H];        // every chunk's per-head weight
};

template <int kSwa>
constexpr size_t smem_bytes() {
  return 1024 + (size_t)Layout<kSwa>::kTileBytes + kQBytes + sizeof(AttnSmem);
}
static_assert(smem_bytes<kMixSwa>() <= 232448, "mixed layout exceeds the shared-memory limit");
static_assert(kRedOff >= (ATTN_CHUNK + kMixSwa) * 128 && kRedOff + 4 * H * 4 <= kQBytes, "reductions overlap P");

// byte offset of 16-byte chunk `c` (0..63 along 512 fp16 channels) of row r in a
// K-major SW128 tile made of 64-channel columns of `col_bytes` each
__device__ __forceinline__ uint32_t swz_off(int r, int c, int col_bytes) {
  return (uint32_t)((c >> 3) * col_bytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

// Butterfly transpose-reduction over the 32 lanes of a warp: on entry every
// lane holds v[0..31] (one value per head column); on exit v[0] of lane l holds
// the reduction over all lanes of column l.
template <bool kMax>
__device__ __forceinline__ void warp_transpose_reduce(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16, n = 32; o >= 1; o >>= 1, n >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      const float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
  }
}

template <int kSwa>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const AttnArgs a) {
  using Lay = Layout<kSwa>;
  constexpr bool kMixed = kSwa > 0;
  constexpr int kAtomCol = Lay::kAtomCol;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *tile = base;                  // [8 cols][rows][128 B] fp16, SW128
  uint8_t *qs = base + Lay::kTileBytes;  // [8 cols][64 heads][128 B] fp16, SW128; later P
  AttnSmem &S = *reinterpret_cast<AttnSmem *>(qs + kQBytes);
  MergeSmem &MS = *reinterpret_cast<MergeSmem *>(tile + H * D * 2);
  float(*red)[H] = reinterpret_cast<float(*)[H]>(qs + kRedOff);   // [4][64]: live only in the softmax

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int chunk = blockIdx.x, p = blockIdx.y;   // p: this launch's problem (block-local)
  const int64_t gp = a.p0 + p;                     // the query token it serves
  const bool is_swa = !kMixed && chunk >= a.n_kchunks;   // split layout: a chunk of SWA rows
  const int64_t seq = gp / a.tokens;
  const int64_t seq_row0 = seq * a.cap;           // the token's sequence in the main-KV cache

  if (tid == 0) {
    mbar_init(&S.bar_load, 1);
    mbar_init(&S.bar_mma, 1);
    mbar_init(&S.bar_ml, 1);
    mbar_init(&S.bar_merge, 1);
    if (a.cluster) {
      // armed before the first cluster barrier, so before any peer's copy
      // into this CTA can start: every other chunk sends its (m, l) record
      // and this CTA's slice of its partial
      const uint32_t crank = cluster_ctarank(), nct = cluster_nctarank();
      const uint32_t slice = ((crank + 1) * kGroups / nct - crank * kGroups / nct) * 128;
      mbar_arrive_expect_tx(&S.bar_ml, (nct - 1) * (2 * H * 4));
      mbar_arrive_expect_tx(&S.bar_merge, (nct - 1) * slice);
    }
    fence_barrier_init();
  }
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;
  bool ok = true;

  // ------------------------------------------------------------------ loads
  // One mbarrier counts the bulk bytes: Q (8 TMA boxes of [64 heads x 64
  // dims] bf16 into the SW128 K-major layout) and the chunk's SWA rows (split:
  // one contiguous copy into the tile's upper half; mixed: 8-row pieces into
  // the SWA-row areas of tile columns 0-3, which the top-K rows never touch).
  // The selected FP4 entries arrive by cp.async into the tile's tail.
  constexpr int kSwaPer = kMixed ? kSwa : ATTN_CHUNK;   // SWA rows per chunk
  constexpr int kSwaRow = kMixed ? ATTN_CHUNK : 0;      // their first tile row
  const int t0 = kMixed ? chunk * kSwa : (chunk - a.n_kchunks) * ATTN_CHUNK;   // first SWA row of this chunk
  int swa_rows = 0;
  int64_t swa_row0 = 0;                              // first SWA row of the token's window
  if (kMixed || is_swa) {
    int len;
    if (a.causal_swa) {
      const int64_t pos = a.first_pos + gp % a.tokens;
      const int64_t start = pos - a.W + 1 > 0 ? pos - a.W + 1 : 0;
      swa_row0 = seq * a.swa_seq_rows + (start - a.swa_first_pos);
      len = (int)(pos - start + 1);
    } else {
      swa_row0 = gp * a.W;
      len = min(__ldg(a.swa_len + gp), a.W);
    }
    swa_rows = max(0, min(kSwaPer, len - t0));
    if (tid < kSwaPer)
      S.row_scale[kSwaRow + tid] = (tid < swa_rows) ? __ldg(a.swa_scale + swa_row0 + t0 + tid) : 0.0f;
  }
  if (!is_swa && tid < ATTN_CHUNK) S.row_scale[tid] = 1.0f;
  if (tid == 0) {
    // Q and the SWA rows first: their latency overlaps the index loads below
    const uint32_t bytes = (uint32_t)kQBytes + (uint32_t)swa_rows * D;
    mbar_arrive_expect_tx(&S.bar_load, bytes);
#pragma unroll
    for (int j = 0; j < D / 64; ++j) tma_load_2d(qs + j * kQAtomCol, &tm_q, j * 64, (int32_t)(gp * H), &S.bar_load);
    if (kMixed) {
      for (int i = 0; i * 8 < swa_rows; ++i)
        bulk_g2s(tile + i * kAtomCol + ATTN_CHUNK * 128, a.swa + (swa_row0 + t0 + 8 * i) * D,
                 (uint32_t)min(8, swa_rows - 8 * i) * D, &S.bar_load);
    } else if (is_swa && swa_rows > 0) {
      bulk_g2s(tile + Lay::kSwaStageOff, a.swa + (swa_row0 + t0) * D, (uint32_t)swa_rows * D, &S.bar_load);
    }
  }
  if (tid < ATTN_CHUNK) {
    bool v;
    if (!is_swa) {
      const int j = chunk * ATTN_CHUNK + tid;
      int32_t id = (j < a.K) ? __ldg(a.idx + gp * a.K + j) : -1;
      if (id >= a.cap) {
        set_error(CSA2_DEV_ERR_INDEX);
        id = -1;
      }
      S.ids[tid] = id;
      v = id >= 0;
    } else {
      v = tid < swa_rows;
    }
    const uint32_t m = __ballot_sync(0xffffffffu, v);
    if (lane == 0) S.vmask[warp] = m;
  } else if (kMixed && warp == ATTN_CHUNK / 32) {
    const uint32_t m = __ballot_sync(0xffffffffu, lane < swa_rows);
    if (lane == 0) S.vmask[warp] = m;
  }
  if (!is_swa) {
    // gather: the selected entries' 288 bytes as 18 16-byte pieces each, all
    // threads issuing their cp.async copies at once
    __syncthreads();
#pragma unroll
    for (int j = 0; j < (ATTN_CHUNK * ENTRY_BYTES / 16) / kThreads; ++j) {
      const int c = tid + j * kThreads;
      const int e = c / (ENTRY_BYTES / 16), piece = c % (ENTRY_BYTES / 16);
      const int32_t id = S.ids[e];
      if (id >= 0)
        cp_async16(tile + Lay::kStageOff + e * ENTRY_BYTES + piece * 16,
                   a.kv + (seq_row0 + id) * ENTRY_BYTES + piece * 16);
    }
    cp_async_commit();
  }
  ok = mbar_wait(&S.bar_load, 0);

  // Q: bf16 -> fp16 in place (same 2-byte slots of the swizzled layout;
  // |q| < 65504 assumed)
#pragma unroll 4
  for (int i = tid; i < kQBytes / 16; i += kThreads) {
    uint4 *ptr = reinterpret_cast<uint4 *>(qs) + i;
    const uint4 v = *ptr;
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint4 o;
    o.x = pack_half2(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u));
    o.y = pack_half2(__uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
    o.z = pack_half2(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u));
    o.w = pack_half2(__uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
    *ptr = o;
  }

  // ---------------------------------------------------------------- dequant
  const int row = tid >> 1, half = tid & 1;   // 2 threads per key, 256 channels each
  if (!is_swa) {
    cp_async_wait_all();
    __syncthreads();   // every thread's gathered pieces have landed
    const bool valid = (S.vmask[row >> 5] >> (row & 31)) & 1;
    uint4 codes[8];
    uint4 scl;
    const uint8_t *src = tile + Lay::kStageOff + row * ENTRY_BYTES;
    if (valid && ok) {
#pragma unroll
      for (int k = 0; k < 8; ++k) codes[k] = *reinterpret_cast<const uint4 *>(src + half * 128 + k * 16);
      scl = *reinterpret_cast<const uint4 *>(src + 256 + half * 16);
    } else {
#pragma unroll
      for (int k = 0; k < 8; ++k) codes[k] = make_uint4(0, 0, 0, 0);
      scl = make_uint4(0, 0, 0, 0);
    }
    // mixed: the 32 SWA rows -- thread (r, j) takes dims 64j..64j+63 of row r
    // from its staging piece (column r / 8, slot r % 8); read now, so that
    // one barrier covers both staging areas
    const int sr = tid >> 3, sj = tid & 7;
    uint4 sraw[4];
    if (kMixed) {
      const bool sv = sr < swa_rows && ok;
      const uint4 *ssrc =
          reinterpret_cast<const uint4 *>(tile + (sr >> 3) * kAtomCol + ATTN_CHUNK * 128 + (sr & 7) * D + sj * 64);
#pragma unroll
      for (int k = 0; k < 4; ++k) sraw[k] = sv ? ssrc[k] : make_uint4(0, 0, 0, 0);
    }
    __syncthreads();   // the staging areas are read; the tile may now be written over them
    const uint32_t sw[4] = {scl.x, scl.y, scl.z, scl.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      // 16 bytes of codes = 32 channels = scale groups 2k, 2k+1 of this half
      const uint32_t cw[4] = {codes[k].x, codes[k].y, codes[k].z, codes[k].w};
#pragma unroll
      for (int g = 0; g < 2; ++g) {
        const uint32_t sb = (sw[k >> 1] >> (8 * ((k & 1) * 2 + g))) & 0xFFu;
        const uint32_t s2 = e4m3x2_to_half2((uint16_t)(sb | (sb << 8)));
        uint32_t h0[4], h1[4];
        e2m1x8_to_half2x4(cw[2 * g], h0);
        e2m1x8_to_half2x4(cw[2 * g + 1], h1);
        uint4 o0, o1;
        o0.x = hmul2_u32(h0[0], s2); o0.y = hmul2_u32(h0[1], s2);
        o0.z = hmul2_u32(h0[2], s2); o0.w = hmul2_u32(h0[3], s2);
        o1.x = hmul2_u32(h1[0], s2); o1.y = hmul2_u32(h1[1], s2);
        o1.z = hmul2_u32(h1[2], s2); o1.w = hmul2_u32(h1[3], s2);
        const int ch16 = half * 32 + k * 4 + g * 2;   // 16-byte chunk index of the first 8 channels
        *reinterpret_cast<uint4 *>(tile + swz_off(row, ch16, kAtomCol)) = o0;
        *reinterpret_cast<uint4 *>(tile + swz_off(row, ch16 + 1, kAtomCol)) = o1;
      }
    }
    if (kMixed) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint32_t w[4] = {sraw[k].x, sraw[k].y, sraw[k].z, sraw[k].w};
        uint4 o0, o1;
        o0.x = e4m3x2_to_half2((uint16_t)(w[0] & 0xFFFF)); o0.y = e4m3x2_to_half2((uint16_t)(w[0] >> 16));
        o0.z = e4m3x2_to_half2((uint16_t)(w[1] & 0xFFFF)); o0.w = e4m3x2_to_half2((uint16_t)(w[1] >> 16));
        o1.x = e4m3x2_to_half2((uint16_t)(w[2] & 0xFFFF)); o1.y = e4m3x2_to_half2((uint16_t)(w[2] >> 16));
        o1.z = e4m3x2_to_half2((uint16_t)(w[3] & 0xFFFF)); o1.w = e4m3x2_to_half2((uint16_t)(w[3] >> 16));
        const int ch16 = sj * 8 + k * 2;
        *reinterpret_cast<uint4 *>(tile + swz_off(ATTN_CHUNK + sr, ch16, kAtomCol)) = o0;
        *reinterpret_cast<uint4 *>(tile + swz_off(ATTN_CHUNK + sr, ch16 + 1, kAtomCol)) = o1;
      }
    }
  } else {
    // SWA rows (E4M3) staged in the tile's upper half: through registers, then
    // converted to fp16 (exact) into the tile
    const bool valid = row < swa_rows && ok;
    uint4 raw[16];
    const uint4 *src = reinterpret_cast<const uint4 *>(tile + Lay::kSwaStageOff + row * D + half * 256);
#pragma unroll
    for (int k = 0; k < 16; ++k) raw[k] = valid ? src[k] : make_uint4(0, 0, 0, 0);
    __syncthreads();   // the staging area is read; the tile may now be written over it
#pragma unroll
    for (int k = 0; k < 16; ++k) {
      const uint32_t w[4] = {raw[k].x, raw[k].y, raw[k].z, raw[k].w};
      uint4 o0, o1;
      o0.x = e4m3x2_to_half2((uint16_t)(w[0] & 0xFFFF)); o0.y = e4m3x2_to_half2((uint16_t)(w[0] >> 16));
      o0.z = e4m3x2_to_half2((uint16_t)(w[1] & 0xFFFF)); o0.w = e4m3x2_to_half2((uint16_t)(w[1] >> 16));
      o1.x = e4m3x2_to_half2((uint16_t)(w[2] & 0xFFFF)); o1.y = e4m3x2_to_half2((uint16_t)(w[2] >> 16));
      o1.z = e4m3x2_to_half2((uint16_t)(w[3] & 0xFFFF)); o1.w = e4m3x2_to_half2((uint16_t)(w[3] >> 16));
      const int ch16 = half * 32 + k * 2;
      *reinterpret_cast<uint4 *>(tile + swz_off(row, ch16, kAtomCol)) = o0;
      *reinterpret_cast<uint4 *>(tile + swz_off(row, ch16 + 1, kAtomCol)) = o1;
    }
  }
  fence_proxy_async_smem();
  __syncthreads();

  // ------------------------------------------------------------- S^T = K Q^T
  if (tid == 0 && ok) {
    tc_fence_after();
    const uint32_t ta = smem_u32(tile), qa = smem_u32(qs);
    // even and odd K steps accumulate into two column blocks, two
    // independent chains that the softmax adds
#pragma unroll 4
    for (int kk = 0; kk < D / 16; ++kk) {
      const uint32_t aa = ta + (kk >> 2) * kAtomCol + (kk & 3) * 32;
      const uint64_t bd = smem_desc(qa + (kk >> 2) * kQAtomCol + (kk & 3) * 32, 16, 1024);
      mma_f16(tmem + (uint32_t)((kk & 1) * H), smem_desc(aa, 16, 1024), bd, kIdescQK, kk > 1 ? 1u : 0u);
      // mixed: the same over tile rows 32..159, whose D lanes 96..127 are the SWA rows
      if (kMixed)
        mma_f16(tmem + (uint32_t)((2 + (kk & 1)) * H), smem_desc(aa + 32 * 128, 16, 1024), bd, kIdescQK,
                kk > 1 ? 1u : 0u);
    }
    mma_commit(&S.bar_mma);
  }
  if (ok) ok = mbar_wait(&S.bar_mma, 0);
  tc_fence_after();

  // ---------------------------------------------------------------- softmax
  // Warp w owns key rows 32 (w % 4) .. + 31 (its TMEM lane quadrant) for heads
  // 32 (w / 4) .. + 31; in the mixed layout warps 3 and 7 also own the SWA
  // rows 128..159 (lanes 96..127 of the second accumulator).
  const int quad = warp & 3, hh = warp >> 2;
  const int key = quad * 32 + lane;
  const bool extra = kMixed && quad == 3;
  const int key2 = ATTN_CHUNK + lane;
  // log2(e) / sqrt(512), times the SWA row scale (the key is code x scale)
  constexpr float kLogit = 0.06375871295460785f;
  float s[32], s2[32];
  {
    uint32_t v[32], v2[32];
    tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(hh * 32), v);
    tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(H + hh * 32), v2);
    tmem_ld_wait();
    const bool valid = ok && ((S.vmask[key >> 5] >> (key & 31)) & 1);
    const float f = kLogit * S.row_scale[key];
#pragma unroll
    for (int i = 0; i < 32; ++i) s[i] = valid ? (__uint_as_float(v[i]) + __uint_as_float(v2[i])) * f : -INFINITY;
  }
  if (extra) {
    uint32_t v[32], v2[32];
    tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(2 * H + hh * 32), v);
    tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(3 * H + hh * 32), v2);
    tmem_ld_wait();
    const bool valid = ok && ((S.vmask[key2 >> 5] >> (key2 & 31)) & 1);
    const float f = kLogit * S.row_scale[key2];
#pragma unroll
    for (int i = 0; i < 32; ++i) s2[i] = valid ? (__uint_as_float(v[i]) + __uint_as_float(v2[i])) * f : -INFINITY;
  }
  {
    float t[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) t[i] = extra ? fmaxf(s[i], s2[i]) : s[i];
    warp_transpose_reduce<true>(t, lane);
    red[quad][hh * 32 + lane] = t[0];
  }
  tc_fence_before();
  __syncthreads();
  if (tid < H) S.mfin[tid] = fmaxf(fmaxf(red[0][tid], red[1][tid]), fmaxf(red[2][tid], red[3][tid]));
  __syncthreads();
  {
    // P = 2^(s - m) per head, times the row scale, as fp16 [rows][64 heads],
    // MN-major SW128 (row r at byte 128 r, 16-byte chunks XOR r % 8)
    float t[32];
    auto write_p = [&](const float(&sv)[32], int k, bool acc) {
      const float rs = S.row_scale[k];
      uint8_t *prow = qs + k * 128;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int i0 = c * 8 + 2 * q;
          const float m0 = S.mfin[hh * 32 + i0], m1 = S.mfin[hh * 32 + i0 + 1];
          const float p0 = (m0 == -INFINITY) ? 0.0f : exp2f(sv[i0] - m0);
          const float p1 = (m1 == -INFINITY) ? 0.0f : exp2f(sv[i0 + 1] - m1);
          t[i0] = acc ? t[i0] + p0 : p0;
          t[i0 + 1] = acc ? t[i0 + 1] + p1 : p1;
          w[q] = pack_half2(p0 * rs, p1 * rs);
        }
        *reinterpret_cast<uint4 *>(prow + (((hh * 4 + c) ^ (k & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    };
    write_p(s, key, false);
    if (extra) write_p(s2, key2, true);
    warp_transpose_reduce<false>(t, lane);
    __syncthreads();   // every thread has read mfin/red before red is reused
    red[quad][hh * 32 + lane] = t[0];
  }
  fence_proxy_async_smem();
  __syncthreads();
  if (tid < H) S.lfin[tid] = (red[0][tid] + red[1][tid]) + (red[2][tid] + red[3][tid]);

  // --------------------------------------------------------------- O = P V
  // P as A, MN-major (heads contiguous): rows 0-63 are the heads, and the
  // second 64-row atom is the same P (leading offset 0), so D lanes 64-127
  // repeat lanes 0-63 and all four TMEM lane quadrants hold heads.  V as B,
  // MN-major: 4 of the tile's 64-dim columns per instruction.  D overwrites S
  // in TMEM (S has been read into registers): lane = head, column = dim.
  if (tid == 0 && ok) {
    tc_fence_after();
    const uint32_t ta = smem_u32(tile), pa = smem_u32(qs);
#pragma unroll
    for (int kk = 0; kk < Lay::kRows / 16; ++kk) {
      const uint64_t ad = smem_desc(pa + kk * 2048, 0, 1024);
#pragma unroll
      for (int nh = 0; nh < D / (int)kPVN; ++nh) {
        const uint64_t bd = smem_desc(ta + (nh * (kPVN / 64)) * kAtomCol + kk * 2048, kAtomCol, 1024);
        mma_f16(tmem + nh * kPVN, ad, bd, kIdescPV, kk > 0 ? 1u : 0u);
      }
    }
    mma_commit(&S.bar_mma);
  }
  if (ok) ok = mbar_wait(&S.bar_mma, 1);
  tc_fence_after();
  const bool all_ok = __syncthreads_and(ok) != 0;

  // Warp w reads TMEM lane quadrant w % 4, i.e. heads 32 (w & 1) + lane; the
  // four warps on the same heads take one quarter of the 512 dims each.
  const int eh = (warp & 1) * 32 + lane;                       // head of this thread's TMEM lane
  const int ec0 = (((warp >> 1) & 1) * 2 + (warp >> 2)) * 128;  // first dim of its quarter
  const uint32_t etm = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)ec0;

  // ---------------------------------------------------------------- merge
  if (a.cluster) {
    // The token's chunks are the CTAs of one cluster.  Each CTA normalises
    // its partial (O / l) into fp16 (a convex combination of values: |.| <=
    // 6 x 448), then pushes to every other CTA, by bulk shared-to-shared
    // copies, its (m, l) record and the slice of the [head][dim] partial that
    // CTA owns.  Each CTA then sums its slice over the chunks with weights
    // l_c 2^(m_c - M) / L straight into the output.
    const uint32_t crank = cluster_ctarank(), nct = cluster_nctarank();
    cluster_arrive();   // this CTA's Q/P region is free to receive
    if (tid < H && !all_ok) {
      S.mfin[tid] = -INFINITY;
      S.lfin[tid] = 0.0f;
    }
    uint8_t *sendb = tile;   // [64 heads][1024 B] fp16, 16-byte chunks XOR-swizzled by (head & 7)
    {
      const float l = S.lfin[eh];
      const float inv = (all_ok && l > 0.0f) ? 1.0f / l : 0.0f;
#pragma unroll 1
      for (int j = 0; j < 4; j += 2) {
        uint32_t v[2][32];
        tmem_ld32(etm + (uint32_t)(j * 32), v[0]);
        tmem_ld32(etm + (uint32_t)(j * 32 + 32), v[1]);
        tmem_ld_wait();
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 o;
            o.x = pack_half2(__uint_as_float(v[u][8 * t + 0]) * inv, __uint_as_float(v[u][8 * t + 1]) * inv);
            o.y = pack_half2(__uint_as_float(v[u][8 * t + 2]) * inv, __uint_as_float(v[u][8 * t + 3]) * inv);
            o.z = pack_half2(__uint_as_float(v[u][8 * t + 4]) * inv, __uint_as_float(v[u][8 * t + 5]) * inv);
            o.w = pack_half2(__uint_as_float(v[u][8 * t + 6]) * inv, __uint_as_float(v[u][8 * t + 7]) * inv);
            const int cr = (ec0 + (j + u) * 32) / 8 + t;   // 16-byte chunk of the head's row
            *reinterpret_cast<uint4 *>(sendb + eh * kRowBytes + (((cr & ~7) | ((cr & 7) ^ (eh & 7))) << 4)) = o;
          }
      }
    }
    fence_proxy_async_smem();   // the bulk copies read what the threads wrote
    __syncthreads();
    cluster_wait();             // every CTA of the cluster may now receive
    if (tid < (int)nct && tid != (int)crank) {
      const uint32_t s = (uint32_t)tid;
      const uint32_t g0 = s * kGroups / nct, bytes = ((s + 1) * kGroups / nct - g0) * 128;
      const uint32_t slot = crank < s ? crank : crank - 1;
      bulk_s2s_cluster(dsmem_addr(&MS.ml_in[crank][0][0], s), S.mfin, 2 * H * 4, dsmem_addr(&S.bar_ml, s));
      bulk_s2s_cluster(dsmem_addr(qs + slot * bytes, s), sendb + g0 * 128, bytes, dsmem_addr(&S.bar_merge, s));
    }
    // warps 0-1 wait for the (m, l) records and compute the weights while
    // warp 2 waits for the partial slices
    if (warp == 2) mbar_wait(&S.bar_merge, 0);
    if (tid < H) {
      mbar_wait(&S.bar_ml, 0);
      float mc[kMaxClusterChunks], lc[kMaxClusterChunks];
      float M = -INFINITY;
#pragma unroll
      for (int c = 0; c < kMaxClusterChunks; ++c)
        if (c < (int)nct) {
          mc[c] = c == (int)crank ? S.mfin[tid] : MS.ml_in[c][0][tid];
          lc[c] = c == (int)crank ? S.lfin[tid] : MS.ml_in[c][1][tid];
          M = fmaxf(M, mc[c]);
        }
      float L = 0.0f;
#pragma unroll
      for (int c = 0; c < kMaxClusterChunks; ++c)
        if (c < (int)nct && mc[c] != -INFINITY) L += lc[c] * exp2f(mc[c] - M);
      const float invL = L > 0.0f ? 1.0f / L : 0.0f;
#pragma unroll
      for (int c = 0; c < kMaxClusterChunks; ++c)
        if (c < (int)nct) MS.wgt[c][tid] = mc[c] == -INFINITY ? 0.0f : lc[c] * exp2f(mc[c] - M) * invL;
      if (crank == 0 && a.lse)
        a.lse[gp * H + tid] = (L > 0.0f) ? (M + log2f(L)) * 0.69314718055994531f : -INFINITY;
    }
    __syncthreads();
    cluster_arrive();   // everything this CTA needs has arrived: its peers' buffers are free
    const uint32_t g0 = crank * kGroups / nct, g1 = (crank + 1) * kGroups / nct;
    const uint32_t bytes = (g1 - g0) * 128;
    float *outp = a.out + gp * H * D;
    for (int k = (int)g0 * 8 + tid; k < (int)g1 * 8; k += kThreads) {
      const int h = k >> 6, cr = k & 63;   // head, 16-byte chunk (8 dims) of its row
      const uint32_t off = (uint32_t)(h * kRowBytes + (((cr & ~7) | ((cr & 7) ^ (h & 7))) << 4));
      float acc[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
#pragma unroll
      for (int c = 0; c < kMaxClusterChunks; ++c)
        if (c < (int)nct) {
          const uint8_t *src = c == (int)crank ? sendb + off
                                               : qs + (uint32_t)(c < (int)crank ? c : c - 1) * bytes + off - g0 * 128;
          const uint4 v = *reinterpret_cast<const uint4 *>(src);
          const float w = MS.wgt[c][h];
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = __half22float2(*reinterpret_cast<const __half2 *>(&u[i]));
            acc[2 * i] = fmaf(w, f.x, acc[2 * i]);
            acc[2 * i + 1] = fmaf(w, f.y, acc[2 * i + 1]);
          }
        }
      float4 *dst = reinterpret_cast<float4 *>(outp + h * D + cr * 8);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    cluster_wait();   // no CTA leaves while a peer's copy may still read its buffer
  } else {
    // unnormalised partial O of this chunk, with its per-head (max, sum), to
    // the workspace for the combine kernel
    const int64_t pc = (int64_t)p * a.n_chunks + chunk;
    {
      float *po = a.part_o + (pc * H + eh) * D + ec0;
#pragma unroll 1
      for (int j = 0; j < 4; ++j) {
        uint32_t v[32];
        tmem_ld32(etm + (uint32_t)(j * 32), v);
        tmem_ld_wait();
#pragma unroll
        for (int t = 0; t < 8; ++t)
          reinterpret_cast<float4 *>(po + j * 32)[t] =
              all_ok ? make_float4(__uint_as_float(v[4 * t]), __uint_as_float(v[4 * t + 1]),
                                   __uint_as_float(v[4 * t + 2]), __uint_as_float(v[4 * t + 3]))
                     : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    if (tid < H) {
      a.part_ml[pc * 2 * H + tid] = all_ok ? S.mfin[tid] : -INFINITY;
      a.part_ml[pc * 2 * H + H + tid] = all_ok ? S.lfin[tid] : 0.0f;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// Merge the chunk partials of each (token, head): m = max_c m_c,
// l = sum_c l_c 2^(m_c - m), o = sum_c o_c 2^(m_c - m) / l; lse in natural log.
__global__ void __launch_bounds__(256) attn_combine_kernel(const AttnArgs a) {
  const int p = blockIdx.y;
  const int h = blockIdx.x;
  const int n = a.n_chunks;
  __shared__ float wgt[64];
  __shared__ float inv_l;
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    for (int c = 0; c < n; ++c) m = fmaxf(m, a.part_ml[((int64_t)p * n + c) * 2 * H + h]);
    float l = 0.0f;
    for (int c = 0; c < n; ++c) {
      const float mc = a.part_ml[((int64_t)p * n + c) * 2 * H + h];
      const float w = (mc == -INFINITY) ? 0.0f : exp2f(mc - m);
      wgt[c] = w;
      l += w * a.part_ml[((int64_t)p * n + c) * 2 * H + H + h];
    }
    inv_l = (l > 0.0f) ? 1.0f / l : 0.0f;
    if (a.lse) a.lse[(a.p0 + p) * H + h] = (l > 0.0f) ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
  }
  __syncthreads();
  for (int d = threadIdx.x; d < D; d += blockDim.x) {
    float acc = 0.0f;
    for (int c = 0; c < n; ++c) acc += wgt[c] * a.part_o[(((int64_t)p * n + c) * H + h) * D + d];
    a.out[((a.p0 + p) * H + h) * D + d] = acc * inv_l;
  }
}

}  // namespace

size_t attn_scratch_bytes(int32_t problems, int32_t K, int32_t W) {
  const int n_chunks = (K + ATTN_CHUNK - 1) / ATTN_CHUNK + (W + ATTN_CHUNK - 1) / ATTN_CHUNK;
  size_t b = (size_t)problems * n_chunks * H * D * 4;
  b = (b + 255) & ~size_t(255);
  b += (size_t)problems * n_chunks * 2 * H * 4;
  return (b + 255) & ~size_t(255);
}

namespace {

template <int kSwa>
cudaError_t launch_layout(const AttnArgs &a, const CUtensorMap &tm_q, cudaStream_t stream, int *launches) {
  constexpr size_t smem = smem_bytes<kSwa>();
  cudaError_t err =
      cudaFuncSetAttribute(sparse_attn_kernel<kSwa>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (err != cudaSuccess) return err;
  if (a.cluster) {
    // one cluster per token: its chunks merge in shared memory
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)a.n_chunks, (unsigned)a.problems, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)a.n_chunks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    err = cudaLaunchKernelEx(&cfg, sparse_attn_kernel<kSwa>, tm_q, a);
    *launches += 1;
    return err;
  }
  sparse_attn_kernel<kSwa><<<dim3(a.n_chunks, a.problems), kThreads, smem, stream>>>(tm_q, a);
  *launches += 1;
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_sparse_attn(AttnArgs a, void *scratch, cudaStream_t stream, int *launches) {
  if (a.problems <= 0) return cudaSuccess;
  const int n_top = (a.K + ATTN_CHUNK - 1) / ATTN_CHUNK;
  const int n_split = n_top + (a.W + ATTN_CHUNK - 1) / ATTN_CHUNK;
  const int n_mixed = max(n_top, (a.W + kMixSwa - 1) / kMixSwa);
  uint8_t *p = static_cast<uint8_t *>(scratch);
  a.part_o = reinterpret_cast<float *>(p);
  size_t off = ((size_t)a.problems * n_split * H * D * 4 + 255) & ~size_t(255);
  a.part_ml = reinterpret_cast<float *>(p + off);
  if (n_split == 0) {
    // no key at all: out = 0, lse = -inf
    cudaError_t e = cudaMemsetAsync(a.out + a.p0 * H * D, 0, (size_t)a.problems * H * D * 4, stream);
    if (e != cudaSuccess || !a.lse) return e;
    a.n_chunks = 0;
    attn_combine_kernel<<<dim3(H, a.problems), 256, 0, stream>>>(a);
    ++*launches;
    return cudaGetLastError();
  }
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  // Streaming (a CTA pipelines whole tokens) once the tokens alone fill the
  // SMs -- it keeps every SM's tensor cores busy without a merge; below that,
  // chunk-parallel (a token's chunks on a cluster of CTAs) for latency.
  if (a.kernel == 2 || (a.kernel == 0 && a.problems >= sms)) {
    const ProfileEvents &pe = profile_events(CSA2_KERNEL_SPARSE_ATTN);
    if (pe.start && (err = record_profile_event(pe.start, stream)) != cudaSuccess) return err;
    err = launch_sparse_attn_stream(a, sms, stream, launches);
    if (err == cudaSuccess && pe.stop) err = record_profile_event(pe.stop, stream);
    return err;
  }
  // The mixed layout (4 chunks for 512 + 128 keys) when the split layout's
  // chunks would not fit in one wave of CTAs (one per SM); the split layout
  // (5 chunks, each less work) otherwise.
  const bool mixed = a.W > 0 && n_mixed < n_split && n_mixed <= kMaxClusterChunks &&
                     (int64_t)a.problems * n_split > (int64_t)sms;
  a.n_chunks = mixed ? n_mixed : n_split;
  a.n_kchunks = mixed ? n_mixed : n_top;
  a.cluster = a.n_chunks <= kMaxClusterChunks ? 1 : 0;
  CUtensorMap tm_q;
  if (!make_tmap_bf16(&tm_q, a.q, D, (a.p0 + a.problems) * H, H)) return cudaErrorInvalidValue;
  const ProfileEvents &pe = profile_events(CSA2_KERNEL_SPARSE_ATTN);
  if (pe.start && (err = record_profile_event(pe.start, stream)) != cudaSuccess) return err;
  err = mixed ? launch_layout<kMixSwa>(a, tm_q, stream, launches) : launch_layout<0>(a, tm_q, stream, launches);
  if (err != cudaSuccess) return err;
  if (pe.stop && (err = record_profile_event(pe.stop, stream)) != cudaSuccess) return err;
  if (!a.cluster) {
    attn_combine_kernel<<<dim3(H, a.problems), 256, 0, stream>>>(a);
    ++*launches;
    err = cudaGetLastError();
  }
  return err;
}

}  // namespace csa2
