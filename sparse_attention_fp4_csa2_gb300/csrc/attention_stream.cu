// Streaming sparse-attention readout: one persistent CTA per query token at a
// time, the token's keys streamed through the tensor cores in chunks of 64.
//
// Same result as the chunk-parallel kernel (attention.cu): one softmax over
// {top-K main-KV entries} U {SWA rows}, logits q_h . k_j / sqrt(512), key =
// value = the dequantised 512-d latent ("DeepSeek-v4.1 Flash: Pushing the
// Limits of KV Cache Compression", sections 3.3.1-3.3.2 and 2.4.4;
// "DeepSeek-V4.1-Flash - Architecture", section 2).  Here the chunks of a
// token are not spread over CTAs and merged; a CTA pipelines them, so that
// dequantisation, the two matrix products and the softmax of consecutive
// chunks overlap and no merge is needed:
//   warp 0        Q of the token by TMA (bf16, 128B-swizzled, 8 boxes);
//   warps 8, 9,   the dequant group: per chunk, the 64 keys' FP4 entries
//   12, 13        (gathered through the index list) or E4M3 SWA rows, read
//                 from global memory into registers one chunk ahead and
//                 written as fp16 into one of two 64-key tiles; per token the
//                 in-place bf16 -> fp16 conversion of Q;
//   warp 1        one thread issues S = Q K^T (M = 128 with the 64 heads in
//                 the upper half, N = 64 keys, K = 512) for chunk c and
//                 O^T += V^T P (M = 4 x 128 dims, N = 64 heads, K = 64 keys)
//                 for chunk c - 1;
//   warps 2, 3,   the softmax: thread = head, warp pair = key half; online
//   10, 11        softmax with a lazily raised reference max (only when a
//                 chunk's max exceeds it by more than 2^8 are the partial
//                 sums and O^T rescaled), P = 2^(s - m) x the SWA row scale
//                 in fp16, MN-major [64 keys x 64 heads];
//   warps 4-7     rescale O^T in TMEM when asked, and per token normalise
//                 it and write out (fp32 [64 heads][512]) and lse.
// Every hand-off is an mbarrier; every wait is bounded, and a timed-out wait
// raises an abort flag that ends all roles.
#include "kernels.cuh"

namespace csa2 {

namespace {

constexpr int kKeys = 64;                     // keys per chunk
constexpr int kTileBytes = kKeys * D * 2;     // 64 KB: [8 columns of 64 dims][64 keys][128 B] fp16
constexpr int kAtomCol = kKeys * 128;         // 8 KB
constexpr int kQBytes = H * D * 2;            // 64 KB: [8 columns][64 heads][128 B] fp16
constexpr int kQAtomCol = H * 128;            // 8 KB
constexpr int kPBytes = kKeys * H * 2;        // 8 KB: [64 keys][64 heads] fp16
constexpr int kWarps = 14;
constexpr int kThreads = kWarps * 32;
constexpr int kDeqThreads = 128;              // warps 8, 9, 12, 13
constexpr int kSmThreads = 128;               // warps 2, 3, 10, 11
constexpr int kEpiThreads = 128;              // warps 4-7
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;                 // S[buf]: columns 64 buf .. (lanes 64..127 = heads)
constexpr uint32_t kColO = 256;               // O^T: columns 256 + 64 mt + head (lanes = dims)
constexpr float kLazy = 8.0f;                 // log2 margin before the reference max is raised
constexpr uint32_t kIdescS = idesc_f16(/*fp16*/ 0, /*A K-major*/ 0, /*B K-major*/ 0, /*N*/ kKeys, /*M*/ 128);
constexpr uint32_t kIdescPV = idesc_f16(/*fp16*/ 0, /*A MN-major*/ 1, /*B MN-major*/ 1, /*N*/ H, /*M*/ 128);

enum : uint32_t { kCmdCorrect = 1, kCmdEpilogue = 2, kCmdExit = 3 };

struct __align__(16) StreamSmem {
  uint64_t q_full, q_ready, q_free;
  uint64_t tile_full[2], tile_free[2];
  uint64_t s_full[2], s_free[2];
  uint64_t red_full[2];
  uint64_t p_full[2];
  uint64_t epi_go, epi_done;
  uint64_t o_full;
  uint32_t tmem_base;
  volatile uint32_t abort;
  uint32_t cmd;
  int32_t cmd_token;
  int32_t cmd_buf;
  uint16_t vm16[2][4];              // [buf][dequant warp]: valid bits of keys 16 w .. 16 w + 15
  float rs[2][kKeys];               // per-key scale: 1 (main entries) or the SWA row scale
  float red[2][2][H];               // [buf][key half][head]: chunk max
  float fac[2][H];                  // [buf][head]: O^T rescale factor of the chunk
  uint32_t flag[2][4];              // [buf][softmax warp]: some head of the warp rescales
  float mfin[H];
  float lpart[2][H];
};

constexpr size_t kSmemBytes = 1024 + 2 * (size_t)kTileBytes + kQBytes + 2 * (size_t)kPBytes + sizeof(StreamSmem);
static_assert(kSmemBytes <= 232448, "streaming attention exceeds the shared-memory limit");

__device__ __forceinline__ uint32_t swz(int r, int c, int col_bytes) {
  return (uint32_t)((c >> 3) * col_bytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_h2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t *>(&h);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}

__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Bounded wait that also ends when another role has aborted.
__device__ __forceinline__ bool wait_bar(StreamSmem &S, uint64_t *bar, uint32_t parity) {
  if (S.abort) return false;
  if (mbar_wait(bar, parity)) return true;
  S.abort = 1;
  return false;
}

// The same for a whole warp, with one outcome for all its lanes.
__device__ __forceinline__ bool warp_wait(StreamSmem &S, uint64_t *bar, uint32_t parity) {
  return __all_sync(0xffffffffu, wait_bar(S, bar, parity));
}

// The SWA rows of token gp: first row and count (as in the chunk-parallel kernel).
__device__ __forceinline__ void swa_range(const AttnArgs &a, int64_t gp, int64_t *row0, int *len) {
  if (a.causal_swa) {
    const int64_t seq = gp / a.tokens;
    const int64_t pos = a.first_pos + gp % a.tokens;
    const int64_t start = pos - a.W + 1 > 0 ? pos - a.W + 1 : 0;
    *row0 = seq * a.swa_seq_rows + (start - a.swa_first_pos);
    *len = (int)(pos - start + 1);
  } else {
    *row0 = gp * a.W;
    *len = min(__ldg(a.swa_len + gp), a.W);
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_attn_stream_kernel(const __grid_constant__ CUtensorMap tm_q, const AttnArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *tiles = base;                         // 2 x 64 KB
  uint8_t *qs = base + 2 * kTileBytes;           // 64 KB; the 8 KB before it is tile 1's tail
  uint8_t *ps = qs + kQBytes;                    // 2 x 8 KB
  StreamSmem &S = *reinterpret_cast<StreamSmem *>(ps + 2 * kPBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n_main = (a.K + kKeys - 1) / kKeys;
  const int n_chunks = n_main + (a.W + kKeys - 1) / kKeys;

  if (tid == 0) {
    mbar_init(&S.q_full, 1);
    mbar_init(&S.q_ready, kDeqThreads);
    mbar_init(&S.q_free, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&S.tile_full[b], kDeqThreads);
      mbar_init(&S.tile_free[b], 1);
      mbar_init(&S.s_full[b], 1);
      mbar_init(&S.s_free[b], kSmThreads);
      mbar_init(&S.red_full[b], kSmThreads);
      mbar_init(&S.p_full[b], kSmThreads);
    }
    mbar_init(&S.epi_go, 1);
    mbar_init(&S.epi_done, kEpiThreads);
    mbar_init(&S.o_full, 1);
    S.abort = 0;
    fence_barrier_init();
    prefetch_tmap(&tm_q);
  }
  if (warp == 0) {
    tmem_alloc(&S.tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = S.tmem_base;

  if (warp == 0) {
    // --------------------------------------------------------------- Q loads
    if (lane == 0) {
      int j = 0;
      for (int p = blockIdx.x; p < a.problems; p += gridDim.x, ++j) {
        if (j > 0 && !wait_bar(S, &S.q_free, (uint32_t)((j - 1) & 1))) break;
        const int64_t gp = a.p0 + p;
        mbar_arrive_expect_tx(&S.q_full, (uint32_t)kQBytes);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) tma_load_2d(qs + c * kQAtomCol, &tm_q, c * 64, (int32_t)(gp * H), &S.q_full);
      }
    }
  } else if (warp == 8 || warp == 9 || warp == 12 || warp == 13) {
    // --------------------------------------------------------------- dequant
    const int dt = (warp == 8 ? 0 : warp == 9 ? 1 : warp == 12 ? 2 : 3) * 32 + lane;   // 0..127
    const int row = dt >> 1, half = dt & 1;    // main entries: 2 threads per key, 256 dims each
    uint32_t g = 0;
    int j = 0;
    bool run = true;
    for (int p = blockIdx.x; run && p < a.problems; p += gridDim.x, ++j) {
      const int64_t gp = a.p0 + p;
      const int64_t seq_row0 = (gp / a.tokens) * a.cap;
      int64_t swa_row0;
      int swa_len;
      swa_range(a, gp, &swa_row0, &swa_len);
      for (int c = 0; c < n_chunks; ++c, ++g) {
        const int b = (int)(g & 1);
        uint8_t *tile = tiles + b * kTileBytes;
        bool valid;
        float scale = 1.0f;
        if (c < n_main) {
          const int k = c * kKeys + row;
          int32_t id = k < a.K ? __ldg(a.idx + gp * a.K + k) : -1;
          if (id >= a.cap) {
            set_error(CSA2_DEV_ERR_INDEX);
            id = -1;
          }
          valid = id >= 0;
          uint4 codes[8], scl;
          if (valid) {
            const uint8_t *src = a.kv + (seq_row0 + id) * ENTRY_BYTES;
#pragma unroll
            for (int q = 0; q < 8; ++q) codes[q] = __ldg(reinterpret_cast<const uint4 *>(src + half * 128 + q * 16));
            scl = __ldg(reinterpret_cast<const uint4 *>(src + 256 + half * 16));
          } else {
#pragma unroll
            for (int q = 0; q < 8; ++q) codes[q] = make_uint4(0, 0, 0, 0);
            scl = make_uint4(0, 0, 0, 0);
          }
          if (g >= 2 && !warp_wait(S, &S.tile_free[b], ((g >> 1) & 1) ^ 1)) { run = false; break; }
          const uint32_t sw[4] = {scl.x, scl.y, scl.z, scl.w};
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t cw[4] = {codes[q].x, codes[q].y, codes[q].z, codes[q].w};
#pragma unroll
            for (int gg = 0; gg < 2; ++gg) {
              const uint32_t sb = (sw[q >> 1] >> (8 * ((q & 1) * 2 + gg))) & 0xFFu;
              const uint32_t s2 = e4m3x2_to_half2((uint16_t)(sb | (sb << 8)));
              uint32_t h0[4], h1[4];
              e2m1x8_to_half2x4(cw[2 * gg], h0);
              e2m1x8_to_half2x4(cw[2 * gg + 1], h1);
              uint4 o0, o1;
              o0.x = hmul2_u32(h0[0], s2); o0.y = hmul2_u32(h0[1], s2);
              o0.z = hmul2_u32(h0[2], s2); o0.w = hmul2_u32(h0[3], s2);
              o1.x = hmul2_u32(h1[0], s2); o1.y = hmul2_u32(h1[1], s2);
              o1.z = hmul2_u32(h1[2], s2); o1.w = hmul2_u32(h1[3], s2);
              const int ch16 = half * 32 + q * 4 + gg * 2;
              *reinterpret_cast<uint4 *>(tile + swz(row, ch16, kAtomCol)) = o0;
              *reinterpret_cast<uint4 *>(tile + swz(row, ch16 + 1, kAtomCol)) = o1;
            }
          }
        } else {
          const int t = (c - n_main) * kKeys + row;   // SWA row of the token's window
          valid = t < swa_len;
          if (g >= 2 && !warp_wait(S, &S.tile_free[b], ((g >> 1) & 1) ^ 1)) { run = false; break; }
          const uint4 *src = reinterpret_cast<const uint4 *>(a.swa + (swa_row0 + t) * D + half * 256);
          if (valid) scale = __ldg(a.swa_scale + swa_row0 + t);
#pragma unroll 4
          for (int q = 0; q < 16; ++q) {
            const uint4 raw = valid ? __ldg(src + q) : make_uint4(0, 0, 0, 0);
            const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
            uint4 o0, o1;
            o0.x = e4m3x2_to_half2((uint16_t)(w[0] & 0xFFFF)); o0.y = e4m3x2_to_half2((uint16_t)(w[0] >> 16));
            o0.z = e4m3x2_to_half2((uint16_t)(w[1] & 0xFFFF)); o0.w = e4m3x2_to_half2((uint16_t)(w[1] >> 16));
            o1.x = e4m3x2_to_half2((uint16_t)(w[2] & 0xFFFF)); o1.y = e4m3x2_to_half2((uint16_t)(w[2] >> 16));
            o1.z = e4m3x2_to_half2((uint16_t)(w[3] & 0xFFFF)); o1.w = e4m3x2_to_half2((uint16_t)(w[3] >> 16));
            const int ch16 = half * 32 + q * 2;
            *reinterpret_cast<uint4 *>(tile + swz(row, ch16, kAtomCol)) = o0;
            *reinterpret_cast<uint4 *>(tile + swz(row, ch16 + 1, kAtomCol)) = o1;
          }
        }
        // this warp's keys are 16 (dt / 32) .. + 15, two lanes each
        const uint32_t m = __ballot_sync(0xffffffffu, valid);
        uint32_t keys = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) keys |= ((m >> (2 * i)) & 1u) << i;
        if (lane == 0) S.vm16[b][dt >> 5] = (uint16_t)keys;
        if (half == 0) S.rs[b][row] = valid ? scale : 0.0f;
        fence_proxy_async_smem();
        mbar_arrive(&S.tile_full[b]);
        if (c == 0) {
          // the token's Q: bf16 -> fp16 in place (|q| < 65504), once it has landed
          if (!warp_wait(S, &S.q_full, (uint32_t)(j & 1))) { run = false; break; }
          for (int i = dt; i < kQBytes / 16; i += kDeqThreads) {
            uint4 *ptr = reinterpret_cast<uint4 *>(qs) + i;
            const uint4 v = *ptr;
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint4 o;
            o.x = pack_h2(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u));
            o.y = pack_h2(__uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
            o.z = pack_h2(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u));
            o.w = pack_h2(__uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
            *ptr = o;
          }
          fence_proxy_async_smem();
          mbar_arrive(&S.q_ready);
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------------- MMA
    // One thread runs an event loop over two cursors: the next chunk whose
    // S = Q K^T can be issued (its tile is written, its S buffer read out,
    // and for a token's first chunk its Q converted) and the next chunk
    // whose O^T += V^T P can be issued (its P written; O^T rescaled first if
    // the softmax raised its reference max; for a token's first chunk, the
    // previous token's epilogue done).  Whichever is ready goes first.
    if (lane == 0) {
      const uint32_t qa = smem_u32(qs);
      const int n_tok = a.problems > (int)blockIdx.x ? (a.problems - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
      const uint32_t total = (uint32_t)n_tok * (uint32_t)n_chunks;
      uint32_t gq = 0, gv = 0;      // next chunk for S, for PV (global chunk counters)
      uint32_t n_cmd = 0;           // commands sent to the epilogue warps
      bool epi_pending = false;     // an epilogue command not yet acknowledged
      bool ok = true;
      uint64_t t_idle = 0;
      auto await_epi = [&]() -> bool {
        if (!epi_pending) return true;
        epi_pending = false;
        const bool r = wait_bar(S, &S.epi_done, (n_cmd - 1) & 1);
        return r;
      };
      auto send = [&](uint32_t cmd, int64_t gp, int b) {
        S.cmd = cmd;
        S.cmd_token = (int32_t)gp;
        S.cmd_buf = b;
        mbar_arrive(&S.epi_go);
        ++n_cmd;
      };
      while (ok && gv < total) {
        bool progress = false;
        // ---- S = Q K^T for chunk gq
        if (gq < total && gq < gv + 2) {
          const int b = (int)(gq & 1);
          const int c = (int)(gq % (uint32_t)n_chunks);
          const uint32_t j = gq / (uint32_t)n_chunks;
          if (mbar_test(&S.tile_full[b], (gq >> 1) & 1) && (c != 0 || mbar_test(&S.q_ready, j & 1)) &&
              (gq < 2 || mbar_test(&S.s_free[b], ((gq >> 1) & 1) ^ 1))) {
            tc_fence_after();
            const uint32_t ta = smem_u32(tiles + b * kTileBytes);
#pragma unroll 4
            for (int kk = 0; kk < D / 16; ++kk) {
              const uint64_t ad = smem_desc(qa + ((kk >> 2) - 1) * kQAtomCol + (kk & 3) * 32, 16, 1024);
              const uint64_t bd = smem_desc(ta + (kk >> 2) * kAtomCol + (kk & 3) * 32, 16, 1024);
              mma_f16(tmem + kColS + b * kKeys, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
            }
            mma_commit(&S.s_full[b]);
            if (c == n_chunks - 1) mma_commit(&S.q_free);
            ++gq;
            progress = true;
          }
        }
        // ---- O^T += V^T P for chunk gv
        if (gv < gq) {
          const int b = (int)(gv & 1);
          const int c = (int)(gv % (uint32_t)n_chunks);
          const int64_t gp = a.p0 + blockIdx.x + (int64_t)(gv / (uint32_t)n_chunks) * gridDim.x;
          if (mbar_test(&S.p_full[b], (gv >> 1) & 1)) {
            if (c == 0 && !await_epi()) { ok = false; break; }   // O^T is read out
            if (c > 0 && (S.flag[b][0] | S.flag[b][1] | S.flag[b][2] | S.flag[b][3])) {
              // O^T must hold every earlier chunk before it is rescaled
              if (!await_epi() || !wait_bar(S, &S.tile_free[(gv - 1) & 1], ((gv - 1) >> 1) & 1)) {
                ok = false;
                break;
              }
              send(kCmdCorrect, gp, b);
              if (!wait_bar(S, &S.epi_done, (n_cmd - 1) & 1)) { ok = false; break; }
            }
            tc_fence_after();
            const uint32_t ta = smem_u32(tiles + b * kTileBytes), pa = smem_u32(ps + b * kPBytes);
#pragma unroll 1
            for (int mt = 0; mt < D / 128; ++mt) {
#pragma unroll
              for (int kk = 0; kk < kKeys / 16; ++kk) {
                const uint64_t ad = smem_desc(ta + (2 * mt) * kAtomCol + kk * 2048, kAtomCol, 1024);
                const uint64_t bd = smem_desc(pa + kk * 2048, 8192, 1024);
                mma_f16(tmem + kColO + mt * H, ad, bd, kIdescPV, (c > 0 || kk > 0) ? 1u : 0u);
              }
            }
            mma_commit(&S.tile_free[b]);
            if (c == n_chunks - 1) {
              mma_commit(&S.o_full);
              send(kCmdEpilogue, gp, 0);
              epi_pending = true;
            }
            ++gv;
            progress = true;
          }
        }
        if (progress) {
          t_idle = 0;
        } else {
          __nanosleep(32);   // leave issue slots to the dequant warps on this scheduler
          if (S.abort) break;
          const uint64_t now = globaltimer_ns();
          if (t_idle == 0) {
            t_idle = now;
          } else if (now - t_idle > kWaitBudgetNs) {
            set_error(CSA2_DEV_ERR_TIMEOUT);
            S.abort = 1;
            break;
          }
        }
      }
      if (ok) await_epi();
      S.cmd = kCmdExit;
      mbar_arrive(&S.epi_go);
    }
  } else if (warp == 2 || warp == 3 || warp == 10 || warp == 11) {
    // --------------------------------------------------------------- softmax
    const int quad = warp & 3;                  // TMEM lane quadrant 2 or 3
    const int h = (quad - 2) * 32 + lane;       // head
    const int kh = warp >= 8 ? 1 : 0;           // key half
    const int slot = (warp & 1) | (kh << 1);    // 0..3
    // log2(e) / sqrt(512)
    constexpr float kLogit = 0.06375871295460785f;
    uint32_t g = 0;
    for (int p = blockIdx.x; p < a.problems; p += gridDim.x) {
      float m_ref = -INFINITY, l = 0.0f;
      bool run = true;
      for (int c = 0; c < n_chunks; ++c, ++g) {
        const int b = (int)(g & 1);
        if (!warp_wait(S, &S.s_full[b], (g >> 1) & 1) || !warp_wait(S, &S.tile_full[b], (g >> 1) & 1)) {
          run = false;
          break;
        }
        tc_fence_after();
        uint32_t v[32];
        tmem_ld32(tmem + ((uint32_t)(quad * 32) << 16) + kColS + b * kKeys + kh * 32, v);
        tmem_ld_wait();
        tc_fence_before();
        mbar_arrive(&S.s_free[b]);
        float s[32], mx = -INFINITY;
        const uint32_t vm = (uint32_t)S.vm16[b][2 * kh] | ((uint32_t)S.vm16[b][2 * kh + 1] << 16);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float x = __uint_as_float(v[i]) * (kLogit * S.rs[b][kh * 32 + i]);
          s[i] = ((vm >> i) & 1) ? x : -INFINITY;
          mx = fmaxf(mx, s[i]);
        }
        S.red[b][kh][h] = mx;
        mbar_arrive(&S.red_full[b]);
        if (!warp_wait(S, &S.red_full[b], (g >> 1) & 1)) { run = false; break; }
        const float mc = fmaxf(S.red[b][0][h], S.red[b][1][h]);
        bool resc = false;
        float f = 1.0f;
        if (m_ref == -INFINITY) {
          m_ref = mc;   // nothing accumulated yet: adopt the chunk's max
        } else if (mc > m_ref + kLazy) {
          f = exp2f(m_ref - mc);
          m_ref = mc;
          l *= f;
          resc = true;
        }
        if (kh == 0) S.fac[b][h] = f;
        const uint32_t any = __ballot_sync(0xffffffffu, resc);
        if (lane == 0) S.flag[b][slot] = any;
        // P buffer b is free once the PV of chunk g - 2 has completed
        if (g >= 2 && !warp_wait(S, &S.tile_free[b], ((g >> 1) & 1) ^ 1)) { run = false; break; }
        uint8_t *pb = ps + b * kPBytes;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int key = kh * 32 + i;
          const float pr = (m_ref == -INFINITY) ? 0.0f : exp2f(s[i] - m_ref);
          l += pr;
          *reinterpret_cast<__half *>(pb + key * 128 + ((((h >> 3) ^ (key & 7)) << 4) | ((h & 7) << 1))) =
              __float2half_rn(pr * S.rs[b][key]);
        }
        if (c == n_chunks - 1) {
          if (kh == 0) S.mfin[h] = m_ref;
          S.lpart[kh][h] = l;
        }
        fence_proxy_async_smem();
        mbar_arrive(&S.p_full[b]);
      }
      if (!run) break;
    }
  } else if (warp >= 4 && warp <= 7) {
    // --------------------------------------------------------------- O^T rescale / epilogue
    const int quad = warp & 3;
    const int et = tid - 4 * 32;              // 0..127
    const uint32_t trow = tmem + ((uint32_t)(quad * 32) << 16) + kColO;
    uint32_t k = 0, nt = 0;
    while (true) {
      if (!warp_wait(S, &S.epi_go, k & 1)) break;
      ++k;
      const uint32_t cmd = S.cmd;
      if (cmd == kCmdExit) break;
      if (cmd == kCmdCorrect) {
        const int b = S.cmd_buf;
        tc_fence_after();
#pragma unroll 1
        for (int mt = 0; mt < D / 128; ++mt) {
#pragma unroll 1
          for (int hb = 0; hb < 2; ++hb) {
            uint32_t v[32];
            tmem_ld32(trow + mt * H + hb * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * S.fac[b][hb * 32 + i]);
            tmem_st32(trow + mt * H + hb * 32, v);
          }
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&S.epi_done);
      } else {
        const int64_t gp = S.cmd_token;
        if (!warp_wait(S, &S.o_full, nt & 1)) break;
        ++nt;
        tc_fence_after();
        float *outp = a.out + gp * H * D;
#pragma unroll 1
        for (int mt = 0; mt < D / 128; ++mt) {
          const int d = mt * 128 + quad * 32 + lane;
#pragma unroll 1
          for (int hb = 0; hb < 2; ++hb) {
            uint32_t v[32];
            tmem_ld32(trow + mt * H + hb * 32, v);
            tmem_ld_wait();
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const int hh = hb * 32 + i;
              const float L = S.lpart[0][hh] + S.lpart[1][hh];
              outp[hh * D + d] = L > 0.0f ? __uint_as_float(v[i]) / L : 0.0f;
            }
          }
        }
        if (et < H && a.lse) {
          const float L = S.lpart[0][et] + S.lpart[1][et];
          a.lse[gp * H + et] = L > 0.0f ? (S.mfin[et] + log2f(L)) * 0.69314718055994531f : -INFINITY;
        }
        tc_fence_before();
        mbar_arrive(&S.epi_done);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_sparse_attn_stream(const AttnArgs &a, int num_sms, cudaStream_t stream, int *launches) {
  if (a.problems <= 0) return cudaSuccess;
  cudaError_t err =
      cudaFuncSetAttribute(sparse_attn_stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (err != cudaSuccess) return err;
  CUtensorMap tm_q;
  if (!make_tmap_bf16(&tm_q, a.q, D, (a.p0 + a.problems) * H, H)) return cudaErrorInvalidValue;
  const int grid = a.problems < num_sms ? a.problems : num_sms;
  sparse_attn_stream_kernel<<<grid, kThreads, kSmemBytes, stream>>>(tm_q, a);
  ++*launches;
  return cudaGetLastError();
}

}  // namespace csa2
