// MXFP4 indexer: the indexer K cache and query in FP4 ("DeepSeek-v4.1 Flash:
// Pushing the Limits of KV Cache Compression", section 2.4.4: quantisation-
// aware training "for the FP4 Indexer Q and K"; section 3.1: a 128-dimensional
// MXFP4 indexer-K entry is 68 B).
//
// Format (OCP Microscaling): a block of 32 dims shares one UE8M0 scale 2^E,
// E = floor(log2(max |x|)) - 2 clamped to [-127, 127] (-127 for an all-zero
// block); elements are E2M1_rne_satfinite(x / 2^E).  The cache is two planes,
// codes [rows][64] (dim 2j in the low nibble of byte j) and scales [rows][4]
// (byte E + 127), so that both stay 16-byte aligned for bulk copies.
//
// The sweep reads 68 B per position instead of 256 B.  Tiles are 256 keys:
// a producer brings a tile's codes (a tensor copy with 64-byte swizzle, so
// that the dequant threads' row reads hit distinct banks) and its scales (a
// bulk copy) into a ring of raw stages; eight dequant warps (a thread per key) turn each key row into
// 128 E5M2 bytes code x 2^(E - Emax), Emax the largest of the row's four
// block exponents, in a 128B-swizzled ring; one thread issues eight
// kind::f8f6f4 MMAs per tile (two halves of 128 keys x K = 4 x 32), D[key][h]
// = K . Q^T with the keys on TMEM lanes and the 32 heads on columns, and four
// epilogue warps take a key per thread: score = 2^Emax_key sum_h wq_h
// ReLU(D[key][h]).  The query is quantised the same way (E5M2 code x
// 2^(E - Emax_h)) with 2^Emax_h folded into wq_h = w_h 2^Emax_h (ReLU commutes
// with a positive factor).
//
// Exactness: E2M1 values have two significant bits, so code x 2^k is an E5M2
// number for k >= -15: every operand is the exact dequantised value while a
// block lies within 2^15 of its row's largest block (rows further apart lose
// their smallest elements); the products and their fp32 sums are those of the
// dequantised MXFP4 values.
#include "pipeline.cuh"

namespace csa2 {

namespace {

constexpr int kKeys = FP4_SWEEP_TILE;                    // keys per tile: two MMA halves of M = 128
constexpr int kRaw = 5;                                  // raw stages
constexpr int kRawCodes = kKeys * DI / 2;                // 16 KB of codes
constexpr int kRawBytes = kRawCodes + kKeys * 4;         // + 1 KB of scales
constexpr int kTiles = 3;                                // E5M2 key tiles
constexpr int kTileBytes = kKeys * DI;                   // 32 KB: [256 rows][128 B], one K-atom wide
constexpr int kHalfKeys = 128;                           // MMA M
constexpr int kQBytes = HI * DI;                         // 4 KB: the 32 head rows (MMA N)
constexpr int kAcc = 2;                                  // TMEM accumulators of 2 x 32 columns
constexpr int kTmemCols = kAcc * 2 * HI;                 // 128
constexpr int kEpiWarps = 4;                             // one per TMEM lane quarter
constexpr int kDeqWarps = 8;                             // a thread per key
constexpr int kDeqThreads = kDeqWarps * 32;
constexpr int kDeqWarp0 = 2 + kEpiWarps;
constexpr int kThreads = (kDeqWarp0 + kDeqWarps) * 32;   // producer, MMA, epilogue, dequant warps
// Row exponents handed from the dequant warps to the epilogue.  Slot
// li % kExpSlots is rewritten only after the epilogue has read it: dequant
// (li + kTiles + kAcc) waits for MMA(li + kAcc) to free its tile, and
// MMA(li + kAcc) waits for the epilogue of li to free their accumulator.
constexpr int kExpSlots = kTiles + kAcc;
constexpr uint32_t kIdesc = idesc_f8f6f4(kFmtE5M2, kFmtE5M2, /*N*/ HI, /*M*/ kHalfKeys);
static_assert(kDeqThreads == kKeys, "one dequant thread per key");
static_assert((kTmemCols & (kTmemCols - 1)) == 0 && kTmemCols <= 512, "TMEM allocation");

struct __align__(8) Fp4Smem {
  uint64_t raw_full[kRaw];
  uint64_t raw_empty[kRaw];
  uint64_t tile_full[kTiles];
  uint64_t tile_empty[kTiles];
  uint64_t exp_full[kExpSlots];
  uint64_t qfull[2];
  uint64_t qempty[2];
  uint64_t accfull[kAcc];
  uint64_t accempty[kAcc];
  uint64_t mma_done;
  uint32_t tmem_base;
  uint32_t abort;
  int8_t row_exp[kExpSlots][kKeys];
};

__device__ __forceinline__ volatile uint32_t &abort_of(Fp4Smem &S) {
  return *reinterpret_cast<volatile uint32_t *>(&S.abort);
}

constexpr size_t kSmemBytes = 1024 + (size_t)kTiles * kTileBytes + 2 * (size_t)kQBytes + (size_t)kRaw * kRawBytes +
                              sizeof(Fp4Smem);
static_assert(kSmemBytes <= 232448, "shared memory per CTA");

__device__ __forceinline__ int32_t clamp_nvis_fp4(const int32_t *n_vis, int b, int64_t n_max) {
  int32_t v = __ldg(n_vis + b);
  if (v < 0 || v > n_max) {
    set_error(CSA2_DEV_ERR_NVIS);
    v = v < 0 ? 0 : (int32_t)n_max;
  }
  return v;
}

// 2^k as a float, k in [-127, 127] (2^-127 is subnormal).
__device__ __forceinline__ float exp2i(int k) {
  return k >= -126 ? __uint_as_float((uint32_t)(k + 127) << 23) : __uint_as_float(0x00400000u);
}

// 2^k (k <= 0) as two fp16: exact down to 2^-24, 0 below.
__device__ __forceinline__ uint32_t exp2_half2(int k) {
  uint32_t h;
  if (k >= -14) h = (uint32_t)(k + 15) << 10;
  else if (k >= -24) h = 1u << (k + 24);
  else h = 0;
  return h | (h << 16);
}

// Eight E2M1 codes (a 32-bit word, element 0 in the low nibble) times 2^k as
// eight E5M2 bytes (lo: elements 0..3, hi: 4..7).  An E5M2 number is the high
// byte of the fp16 of the same value (same exponent field, two mantissa
// bits); code x 2^k has two significant bits, so the high byte is exact while
// the value is an E5M2 number (k >= -15).
__device__ __forceinline__ void e2m1x8_to_e5m2x8(uint32_t codes, uint32_t s2, uint32_t &lo, uint32_t &hi) {
  uint32_t h[4];
  e2m1x8_to_half2x4(codes, h);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = hmul2_u32(h[i], s2);
  lo = __byte_perm(h[0], h[1], 0x7531);
  hi = __byte_perm(h[2], h[3], 0x7531);
}

// MXFP4 of one 128-dim row held by a warp, 4 dims per lane (lane l: dims
// 4l..4l+3, block l / 8).  Returns the lane's two code bytes and its block's E.
// (Finite inputs; a subnormal block maximum gives E = -127 like zero does.)
__device__ __forceinline__ uint32_t mxfp4_lane(const float (&x)[4], int *E_out) {
  float am = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
  am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
  const int ef = (int)((__float_as_uint(am) >> 23) & 0xFFu);
  int E = -127;
  if (am > 0.0f && ef > 0) E = max(-127, min(127, ef - 127 - 2));
  const float inv = exp2i(-E);   // x / 2^E, exact
  const uint32_t lo = cvt_e2m1x2(x[1] * inv, x[0] * inv);
  const uint32_t hi = cvt_e2m1x2(x[3] * inv, x[2] * inv);
  *E_out = E;
  return (lo & 0xFFu) | ((hi & 0xFFu) << 8);
}

__device__ __forceinline__ void load_bf16x4(const __nv_bfloat16 *p, float (&x)[4]) {
  const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
  x[0] = __uint_as_float(v.x << 16);
  x[1] = __uint_as_float(v.x & 0xFFFF0000u);
  x[2] = __uint_as_float(v.y << 16);
  x[3] = __uint_as_float(v.y & 0xFFFF0000u);
}

// One warp per row: bf16 [n][128] -> the MXFP4 planes at row slot[i].
__global__ void __launch_bounds__(256) indexer_k_quant_kernel(const __nv_bfloat16 *__restrict__ k, int64_t n,
                                                              const int64_t *__restrict__ slot,
                                                              uint8_t *__restrict__ planes, int64_t rows) {
  pdl_wait();   // the inputs' producer is complete past here (programmatic launch)
  const int lane = threadIdx.x & 31;
  const int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= n) return;   // warp-uniform
  const int64_t row = __ldg(slot + i);
  if (row < 0 || row >= rows) {
    if (lane == 0) set_error(CSA2_DEV_ERR_INDEX);
    return;
  }
  float x[4];
  load_bf16x4(k + i * DI + lane * 4, x);
  int E;
  const uint32_t codes = mxfp4_lane(x, &E);
  reinterpret_cast<uint16_t *>(planes + row * (DI / 2))[lane] = (uint16_t)codes;
  if ((lane & 7) == 0) planes[rows * (DI / 2) + row * 4 + (lane >> 3)] = (uint8_t)(E + 127);
}

// One warp per query row (batch b, head h): bf16 [rows][128] -> its MXFP4
// values as E5M2 bytes code x 2^(E - Emax), and wq = w x 2^Emax.
__global__ void __launch_bounds__(256) indexer_q_fp4_kernel(const __nv_bfloat16 *__restrict__ q,
                                                            const float *__restrict__ w, int64_t rows,
                                                            uint8_t *__restrict__ out, float *__restrict__ wq) {
  pdl_wait();   // the inputs' producer is complete past here (programmatic launch)
  const int lane = threadIdx.x & 31;
  const int64_t i = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (i >= rows) return;
  float x[4];
  load_bf16x4(q + i * DI + lane * 4, x);
  int E;
  const uint32_t codes = mxfp4_lane(x, &E);
  const int emax = max(E, max(__shfl_xor_sync(0xffffffffu, E, 8),
                              max(__shfl_xor_sync(0xffffffffu, E, 16), __shfl_xor_sync(0xffffffffu, E, 24))));
  uint32_t lo, hi;
  e2m1x8_to_e5m2x8(codes, exp2_half2(E - emax), lo, hi);   // the lane's 4 codes -> lo
  reinterpret_cast<uint32_t *>(out + i * DI)[lane] = lo;
  if (lane == 0) wq[i] = __ldg(w + i) * exp2i(emax);
}

// The largest block exponent of a row from its four scale bytes.
__device__ __forceinline__ int row_emax(uint32_t sc) {
  const uint32_t m = __vmaxu4(sc, sc >> 16);
  return (int)max(m & 0xFFu, (m >> 8) & 0xFFu) - 127;
}

template <bool kPool>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_sweep_fp4_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_q,
                             const SweepArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *tiles = base;                                    // kTiles x 32 KB, 1024-aligned
  uint8_t *qbuf = tiles + (size_t)kTiles * kTileBytes;      // 2 x 4 KB
  uint8_t *raw = qbuf + 2 * kQBytes;                        // kRaw x 17 KB
  Fp4Smem &S = *reinterpret_cast<Fp4Smem *>(raw + (size_t)kRaw * kRawBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t total = (int64_t)a.batch * a.tiles_per_seq;
  const int64_t it0 = total * blockIdx.x / gridDim.x;
  const int n_tiles = (int)(total * (blockIdx.x + 1) / gridDim.x - it0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kRaw; ++s) {
      mbar_init(&S.raw_full[s], 1);
      mbar_init(&S.raw_empty[s], kDeqThreads);
    }
    for (int s = 0; s < kTiles; ++s) {
      mbar_init(&S.tile_full[s], kDeqThreads);
      mbar_init(&S.tile_empty[s], 1);
    }
    for (int s = 0; s < kExpSlots; ++s) mbar_init(&S.exp_full[s], kDeqThreads);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&S.qfull[i], 1);
      mbar_init(&S.qempty[i], 1);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(&S.accfull[i], 1);
      mbar_init(&S.accempty[i], kEpiWarps * 32);
    }
    mbar_init(&S.mma_done, 1);
    abort_of(S) = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_q);
  }
  // the inputs' producer is complete past here (programmatic launch)
  pdl_wait();
  if (warp == 1) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // Full tiles: lane 0 alone runs the producer; pool tiles: the whole warp
    if (kPool || lane == 0) {
      // ------------------------------------------------------------ producer
      // lane 0 drives the rings and copies a Full tile: one tensor copy of the
      // tile's code rows (zero-filled past the last row, counted in full) and
      // one bulk copy of its scales; in a pool tile (Reindex) lane j fetches
      // pool block j, its 8 code rows and its scales.  Scale copies are cut to
      // the rows the planes hold.
      const uint64_t pol = l2_policy_evict_first();   // codes are read once
      int prev_b = -1, q_issued = 0;
      int32_t nv = 0;
      int n_issued = 0;
      TileCursor cur(it0, a.tiles_per_seq);
      Ring<kRaw> rr;
      for (int li = 0; li < n_tiles; ++li, cur.next(), rr.next()) {
        const int b = cur.b, t = cur.t;
        int ok = 1;
        if (b != prev_b) {
          if (lane == 0) {
            const int qs = q_issued & 1;
            if (q_issued > 0 && abort_of(S)) {
              ok = 0;
            } else if (!mbar_wait(&S.qempty[qs], ((q_issued >> 1) & 1) ^ 1)) {
              abort_of(S) = 1;
              ok = 0;
            } else {
              mbar_arrive_expect_tx(&S.qfull[qs], kQBytes);
              tma_load_2d(qbuf + qs * kQBytes, &tm_q, 0, b * HI, &S.qfull[qs]);
              nv = clamp_nvis_fp4(a.n_vis, b, a.n_max);
            }
          }
          if (!warp_bcast<kPool>(ok)) break;
          nv = warp_bcast<kPool>(nv);
          ++q_issued;
          prev_b = b;
        }
        const int s = rr.slot;
        if (lane == 0 && !mbar_wait(&S.raw_empty[s], rr.phase ^ 1)) {
          abort_of(S) = 1;
          ok = 0;
        }
        if (!warp_bcast<kPool>(ok)) break;
        uint8_t *dst = raw + (size_t)s * kRawBytes;
        const int64_t row0 = (int64_t)b * a.cap;
        if (!kPool) {
          if (lane == 0) {
            if ((int64_t)t * kKeys < nv) {
              const int64_t r0 = row0 + (int64_t)t * kKeys;
              const int64_t left = a.k_rows - r0;
              const uint32_t nrows = (uint32_t)(left < kKeys ? left : kKeys);   // a multiple of 4
              mbar_arrive_expect_tx(&S.raw_full[s], kRawCodes + nrows * 4);
              tma_load_2d_hint(dst, &tm_k, 0, (int32_t)r0, &S.raw_full[s], pol);
              bulk_g2s(dst + kRawCodes, a.k_scales + r0 * 4, nrows * 4, &S.raw_full[s]);
            } else {
              mbar_arrive(&S.raw_full[s]);
            }
          }
        } else {
          // the tile's pool blocks j0 .. j0 + nj - 1 (the last tile may hold fewer)
          const int64_t j0 = (int64_t)t * (kKeys / BLOCK);
          const int nj = (int)(a.pool_nb - j0 < kKeys / BLOCK ? a.pool_nb - j0 : kKeys / BLOCK);
          const int64_t nblk_vis = ((int64_t)nv + BLOCK - 1) / BLOCK;
          const int32_t blk = lane < nj ? __ldg(a.pool + (int64_t)b * a.pool_nb + j0 + lane) : -1;
          const bool v = blk >= 0 && blk < nblk_vis;
          if (lane < nj && !v && blk >= nblk_vis && (int64_t)blk * BLOCK >= a.n_max) set_error(CSA2_DEV_ERR_POOL);
          const int64_t y = row0 + (int64_t)blk * BLOCK;
          // a block past the last row when cap is not a multiple of 8 (cap and
          // y are multiples of 4)
          const uint32_t nrows = v ? (uint32_t)(a.k_rows - y < BLOCK ? a.k_rows - y : BLOCK) : 0u;
          const uint32_t bytes = __reduce_add_sync(0xffffffffu, v ? BLOCK * (DI / 2) + nrows * 4 : 0u);
          if (bytes) {
            if (lane == 0) mbar_arrive_expect_tx(&S.raw_full[s], bytes);
            __syncwarp();
            if (v) {
              tma_load_2d_hint(dst + lane * BLOCK * (DI / 2), &tm_k, 0, (int32_t)y, &S.raw_full[s], pol);
              bulk_g2s(dst + kRawCodes + lane * BLOCK * 4, a.k_scales + y * 4, nrows * 4, &S.raw_full[s]);
            }
          } else if (lane == 0) {
            mbar_arrive(&S.raw_full[s]);
          }
        }
        ++n_issued;
      }
      // every copy this warp issued has landed before the CTA can exit
      if (lane == 0) {
        for (int s = 0; s < kRaw && s < n_issued; ++s) {
          const int last = s + ((n_issued - 1 - s) / kRaw) * kRaw;
          mbar_wait(&S.raw_full[s], (uint32_t)((last / kRaw) & 1));
        }
        if (q_issued > 0) mbar_wait(&S.qfull[(q_issued - 1) & 1], ((q_issued - 1) >> 1) & 1);
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int prev_b = -1, qi = -1;
      const uint32_t tbase = smem_u32(tiles), qbase = smem_u32(qbuf);
      TileCursor cur(it0, a.tiles_per_seq);
      Ring<kTiles> tr;
      Ring<kAcc> ar;
      for (int li = 0; li < n_tiles; ++li, cur.next(), tr.next(), ar.next()) {
        if (abort_of(S)) break;
        const int b = cur.b;
        if (b != prev_b) {
          if (qi >= 0) mma_commit(&S.qempty[qi & 1]);
          ++qi;
          if (!mbar_wait(&S.qfull[qi & 1], (qi >> 1) & 1)) { abort_of(S) = 1; break; }
          prev_b = b;
        }
        const int st = tr.slot, acc = ar.slot;
        if (!mbar_wait(&S.tile_full[st], tr.phase)) { abort_of(S) = 1; break; }
        if (!mbar_wait(&S.accempty[acc], ar.phase ^ 1)) { abort_of(S) = 1; break; }
        tc_fence_after();
        const uint32_t ka = tbase + (uint32_t)st * kTileBytes;
        const uint32_t qa = qbase + (uint32_t)(qi & 1) * kQBytes;
#pragma unroll
        for (int j = 0; j < 2; ++j)              // keys 128j .. 128j + 127 -> columns 32j .. 32j + 31
#pragma unroll
          for (int kk = 0; kk < DI / 32; ++kk)   // K = 32 E5M2 (32 B) per MMA
            mma_f8f6f4(tmem + (uint32_t)(acc * 2 * HI + j * HI), smem_desc(ka + j * kHalfKeys * DI + kk * 32, 16, 1024),
                       smem_desc(qa + kk * 32, 16, 1024), kIdesc, kk > 0 ? 1u : 0u);
        mma_commit(&S.tile_empty[st]);
        mma_commit(&S.accfull[acc]);
      }
      pdl_release();   // the last tile's MMAs are issued: the next kernel's CTAs may be dispatched
      mma_commit(&S.mma_done);
      mbar_wait(&S.mma_done, 0);
    }
  } else if (warp >= kDeqWarp0) {
    // ------------------------------------------------------------ dequant
    // thread = key row of the tile: 64 code bytes + 4 scale bytes -> 128
    // E5M2 bytes code x 2^(E - Emax); Emax goes to the epilogue
    const int r = threadIdx.x - kDeqWarp0 * 32;   // 0..255
    Ring<kRaw> rr;
    Ring<kTiles> tr;
    Ring<kExpSlots> er;
    for (int li = 0; li < n_tiles; ++li, rr.next(), tr.next(), er.next()) {
      if (abort_of(S)) break;
      const int s = rr.slot, st = tr.slot;
      if (!mbar_wait(&S.raw_full[s], rr.phase)) { abort_of(S) = 1; break; }
      const uint8_t *src = raw + (size_t)s * kRawBytes;
      // block q of the row: 16-byte chunk q ^ ((r >> 1) & 3) (64B swizzle)
      uint4 c[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        c[q] = *reinterpret_cast<const uint4 *>(src + r * (DI / 2) + ((q ^ ((r >> 1) & 3)) << 4));
      const uint32_t sc = *reinterpret_cast<const uint32_t *>(src + kRawCodes + r * 4);
      mbar_arrive(&S.raw_empty[s]);
      const int emax = row_emax(sc);
      if (!mbar_wait(&S.tile_empty[st], tr.phase ^ 1)) { abort_of(S) = 1; break; }
      S.row_exp[er.slot][r] = (int8_t)emax;
      uint8_t *row = tiles + (size_t)st * kTileBytes + r * DI;
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) {   // block bb: 32 codes -> 32 bytes = 16-byte chunks 2bb, 2bb + 1
        const uint32_t s2 = exp2_half2((int)((sc >> (8 * bb)) & 0xFFu) - 127 - emax);
        uint4 o0, o1;
        e2m1x8_to_e5m2x8(c[bb].x, s2, o0.x, o0.y);
        e2m1x8_to_e5m2x8(c[bb].y, s2, o0.z, o0.w);
        e2m1x8_to_e5m2x8(c[bb].z, s2, o1.x, o1.y);
        e2m1x8_to_e5m2x8(c[bb].w, s2, o1.z, o1.w);
        *reinterpret_cast<uint4 *>(row + (((2 * bb) ^ (r & 7)) << 4)) = o0;
        *reinterpret_cast<uint4 *>(row + (((2 * bb + 1) ^ (r & 7)) << 4)) = o1;
      }
      fence_proxy_async_smem();
      mbar_arrive(&S.tile_full[st]);
      mbar_arrive(&S.exp_full[er.slot]);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warp = TMEM lane quarter q: keys 32q + lane and 128 + 32q + lane
    const int quad = warp & 3;
    int prev_b = -1;
    int32_t nv = 0;
    float wv[HI];
    TileCursor cur(it0, a.tiles_per_seq);
    Ring<kAcc> ar;
    Ring<kExpSlots> er;
    for (int li = 0; li < n_tiles; ++li, cur.next(), ar.next(), er.next()) {
      if (abort_of(S)) break;
      const int b = cur.b, t = cur.t;
      if (b != prev_b) {
#pragma unroll
        for (int h = 0; h < HI; ++h) wv[h] = __ldg(a.w + (int64_t)b * HI + h);
        nv = clamp_nvis_fp4(a.n_vis, b, a.n_max);
        prev_b = b;
      }
      const int acc = ar.slot;
      if (!mbar_wait(&S.exp_full[er.slot], er.phase)) { abort_of(S) = 1; break; }
      const int k0 = quad * 32 + lane;
      const float f0 = exp2i(S.row_exp[er.slot][k0]), f1 = exp2i(S.row_exp[er.slot][kHalfKeys + k0]);
      if (!mbar_wait(&S.accfull[acc], ar.phase)) { abort_of(S) = 1; break; }
      tc_fence_after();
      uint32_t v0[32], v1[32];
      const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16) + (uint32_t)(acc * 2 * HI);
      tmem_ld32(taddr, v0);
      tmem_ld32(taddr + HI, v1);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&S.accempty[acc]);
      // sum_h w_h ReLU(.) for the two keys, as two partial sums each (even
      // and odd heads) on the packed fp32 pipe
      uint64_t p0 = 0ull, p1 = 0ull;
#pragma unroll
      for (int h = 0; h < HI; h += 2) {
        const uint64_t w2 = f32x2_pack(wv[h], wv[h + 1]);
        p0 = f32x2_fma(w2, f32x2_pack(fmaxf(__uint_as_float(v0[h]), 0.0f), fmaxf(__uint_as_float(v0[h + 1]), 0.0f)),
                       p0);
        p1 = f32x2_fma(w2, f32x2_pack(fmaxf(__uint_as_float(v1[h]), 0.0f), fmaxf(__uint_as_float(v1[h + 1]), 0.0f)),
                       p1);
      }
      float e0, o0, e1, o1;
      f32x2_unpack(p0, e0, o0);
      f32x2_unpack(p1, e1, o1);
      const float s0 = e0 + o0, s1 = e1 + o1;
      float *srow = a.scores + (int64_t)b * a.row_len;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const float sc = (j ? s1 : s0) * (j ? f1 : f0);
        const int64_t slot = (int64_t)t * kKeys + j * kHalfKeys + k0;
        if (!kPool) {
          const bool ok = slot < nv;
          const float o = ok ? sc : -INFINITY;
          srow[slot] = o;
          if (a.block_scores) {
            // lanes 8i..8i+7 hold the keys of block slot / 8
            float bv;
            if (a.block_reduce == 0) {
              bv = o;
              bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, 1));
              bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, 2));
              bv = fmaxf(bv, __shfl_xor_sync(0xffffffffu, bv, 4));
            } else {
              bv = ok ? sc : 0.0f;
              bv += __shfl_xor_sync(0xffffffffu, bv, 1);
              bv += __shfl_xor_sync(0xffffffffu, bv, 2);
              bv += __shfl_xor_sync(0xffffffffu, bv, 4);
              if ((slot & ~int64_t(BLOCK - 1)) >= nv) bv = -INFINITY;
            }
            const int64_t blk = slot / BLOCK;
            if ((lane & 7) == 0 && blk < a.nblk_stride) a.block_scores[(int64_t)b * a.nblk_stride + blk] = bv;
          }
        } else if (slot < a.row_len) {   // pool_nb * 8 slots
          const int32_t blk = __ldg(a.pool + (int64_t)b * a.pool_nb + slot / BLOCK);
          const int64_t pos = (int64_t)blk * BLOCK + (slot & (BLOCK - 1));
          srow[slot] = (blk >= 0 && pos < nv) ? sc : -INFINITY;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_indexer_k_quant(const void *k, int64_t n, const int64_t *slot, uint8_t *k_fp4, int64_t rows,
                                   cudaStream_t stream) {
  if (n <= 0) return cudaSuccess;
  const int warps = 8;
  return launch_pdl(indexer_k_quant_kernel, dim3((unsigned)((n + warps - 1) / warps)), dim3(warps * 32), 0, stream,
                    0u, static_cast<const __nv_bfloat16 *>(k), n, slot, k_fp4, rows);
}

cudaError_t launch_indexer_q_fp4(const void *q, const float *w, int64_t rows, void *q_e5m2, float *wq,
                                 cudaStream_t stream) {
  if (rows <= 0) return cudaSuccess;
  const int warps = 8;
  return launch_pdl(indexer_q_fp4_kernel, dim3((unsigned)((rows + warps - 1) / warps)), dim3(warps * 32), 0,
                    stream, 0u, static_cast<const __nv_bfloat16 *>(q), w, rows, static_cast<uint8_t *>(q_e5m2), wq);
}

cudaError_t launch_indexer_sweep_fp4(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const SweepArgs &a,
                                     int num_sms, cudaStream_t stream, int *launches) {
  const int64_t total = (int64_t)a.batch * a.tiles_per_seq;
  if (total <= 0) return cudaSuccess;
  const int grid = (int)(total < num_sms ? total : num_sms);
  const ProfileEvents &pe = profile_events(CSA2_KERNEL_INDEXER_SWEEP);
  cudaError_t err;
  if (pe.start && (err = record_profile_event(pe.start, stream)) != cudaSuccess) return err;
  if (a.pool) {
    err = cudaFuncSetAttribute(indexer_sweep_fp4_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    err = launch_pdl(indexer_sweep_fp4_kernel<true>, dim3(grid), dim3(kThreads), kSmemBytes, stream, 0u, tm_k, tm_q,
                     a);
  } else {
    err = cudaFuncSetAttribute(indexer_sweep_fp4_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)kSmemBytes);
    if (err != cudaSuccess) return err;
    err = launch_pdl(indexer_sweep_fp4_kernel<false>, dim3(grid), dim3(kThreads), kSmemBytes, stream, 0u, tm_k, tm_q,
                     a);
  }
  if (err != cudaSuccess) return err;
  ++*launches;
  if (pe.stop) err = record_profile_event(pe.stop, stream);
  return err;
}

}  // namespace csa2
