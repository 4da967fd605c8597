// Shared constants and launcher declarations of the CSA2 kernels.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>

#include "ptx.cuh"

namespace csa2 {

// Head geometry ("DeepSeek-V4.1-Flash - Architecture", section 2, main
// attention settings): 512-d latent with a 64-channel RoPE tail, 64 query
// heads, 32 indexer heads x 128.
constexpr int D = 512;
constexpr int ROPE_DIM = 64;
constexpr int H = 64;
constexpr int HI = 32;
constexpr int DI = 128;
constexpr int ENTRY_BYTES = 288;   // 256 B codes + 32 B E4M3 scales
constexpr int BLOCK = 8;           // HSI candidate block width

// Indexer sweep: 128 positions per tile (the MMA M dimension).
constexpr int SWEEP_TILE = 128;
constexpr int FP4_SWEEP_TILE = 256;   // keys per tile of the MXFP4 sweep
// Radix select: 11-bit first digit.
constexpr int TOPK_BINS = 2048;
constexpr int TOPK_MAX_K = 8192;
// Score histogram of each row, handed from an indexer sweep to the cluster
// top-K of the same call: the row's valid scores counted by the top
// TOPK_HIST_BITS bits of their keys (topk_score_key).  The sweep adds to it,
// the top-K reads it and leaves it zero for the next call.
constexpr int TOPK_HIST_BITS = 12;
constexpr int TOPK_HIST_BINS = 1 << TOPK_HIST_BITS;

// Per-row scratch of a top-K selection (kept in the caller's workspace).
struct TopkScratch {
  uint32_t *hist;      // [rows][TOPK_BINS]
  uint32_t *counters;  // [rows][4]: selected, candidates, threshold bin + 1, above
  int32_t *sel;        // [rows][k]
  uint64_t *cand;      // [rows][row_len]
};

// Description of one batched top-K: rows of `row_len` fp32 values where -inf
// marks an invalid slot.
struct TopkRows {
  const float *vals;       // [rows][row_stride]
  int64_t row_len;
  int64_t row_stride;
  int32_t rows;
  int32_t k;
  // HSI: the block holding position n_vis[b]-1 is forced in (key of +inf)
  const int32_t *force_nvis;  // NULL = no forcing
  int32_t force_block;        // block width for the forced element
  int64_t n_max;              // n_vis clamp
  // output mapping: NULL -> index itself; else slot j -> pool[b][j/8]*8 + j%8
  const int32_t *pool;
  int32_t pool_stride;
  int32_t *out;             // [rows][k] ascending, -1 padded
  // [rows][TOPK_HIST_BINS] histogram of the rows from the sweep that wrote
  // them, or NULL; the cluster top-K starts from it and clears it
  uint32_t *hist = nullptr;
};

// Benchmark timing hook (csa2_set_profile_events): events recorded around a kernel.
struct ProfileEvents {
  cudaEvent_t start = nullptr, stop = nullptr;
};
ProfileEvents &profile_events(int kernel);
// Kernel launches of the last successful call on this host thread
// (csa2_last_launch_count); every entry point sets it.
void set_last_launch_count(int32_t n);
// Records `ev` on `stream`; inside a stream capture it becomes an event-record
// node of the graph, so every replay records it.
cudaError_t record_profile_event(cudaEvent_t ev, cudaStream_t stream);

// Launches `kern` with programmatic stream serialisation (the kernel enters
// through pdl_enter / pdl_wait before touching global memory) and, when
// cluster_x > 0, thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              unsigned cluster_x, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (cluster_x > 0) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// 2-D bf16 tensor map over rows of `inner` elements, box {64, box_rows}, 128B swizzle.
bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t inner, int64_t rows, uint32_t box_rows);

// w_ik != NULL: also the entry's indexer key k = W_ik e into k_out (bf16 rows,
// or the MXFP4 planes with fp4), row slot[i] of k_rows.
cudaError_t launch_kv_quant_write(const void *latent, const void *z, int m, int64_t n_entries, const int64_t *pos,
                                  const int64_t *slot, uint8_t *kv, int64_t kv_rows, float rope_theta,
                                  cudaStream_t stream, const void *w_ik = nullptr, void *k_out = nullptr,
                                  int64_t k_rows = 0, int fp4 = 0);

struct SweepArgs {
  const float *w;             // [B][32]
  const int32_t *n_vis;       // [B]
  const int32_t *pool;        // [B][pool_nb] (Reindex) or NULL (Full)
  float *scores;              // [B][row_len]
  float *block_scores;        // [B][nblk_stride] or NULL
  int64_t cap;
  int64_t n_max;
  int64_t row_len;            // tiles_per_seq * 128
  int32_t batch;
  int32_t tiles_per_seq;
  int32_t pool_nb;
  int32_t nblk_stride;        // ceil(n_max / 8)
  int32_t block_reduce;       // 0 max, 1 sum
  const uint8_t *k_scales;    // MXFP4 sweep: the scale plane [k_rows][4]
  int64_t k_rows;             // MXFP4 sweep: rows of the planes (batch * cap)
  uint32_t *hist = nullptr;   // [B][TOPK_HIST_BINS] (zero on entry) or NULL: every score's key counted
};

cudaError_t launch_indexer_sweep(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const SweepArgs &a,
                                 int num_sms, cudaStream_t stream, int *launches);
// MXFP4 indexer: tm_k over the code plane (bytes [k_rows][64], 64B swizzle,
// boxes of FP4_SWEEP_TILE rows, or of 8 rows for a pool), the scales through
// a.k_scales, tm_q over the queries' E5M2 rows (bytes [batch * 32][128], 128B
// swizzle, boxes of 32 rows).
cudaError_t launch_indexer_sweep_fp4(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const SweepArgs &a,
                                     int num_sms, cudaStream_t stream, int *launches);
cudaError_t launch_indexer_k_quant(const void *k, int64_t n, const int64_t *slot, uint8_t *k_fp4, int64_t rows,
                                   cudaStream_t stream);
// The queries' MXFP4 values as E5M2 bytes [rows][128] (code x 2^(E - Emax) per
// row) and wq = w x 2^Emax.
cudaError_t launch_indexer_q_fp4(const void *q, const float *w, int64_t rows, void *q_e5m2, float *wq,
                                 cudaStream_t stream);

// Single-kernel top-K with one thread-block cluster per row (no scratch);
// for k <= 2048.
bool topk_cluster_supported(const TopkRows &r);
// profiled: record the CSA2_KERNEL_TOPK events (the indexer's top-K), not for
// the HSI pool selection.
cudaError_t launch_topk_cluster(const TopkRows &r, cudaStream_t stream, int *launches, bool profiled = true);

// Single-kernel top-K with one CTA per row, for rows of at most 131,072
// scores and k <= 2048.
bool topk_row_supported(const TopkRows &r);
cudaError_t launch_topk_row(const TopkRows &r, cudaStream_t stream, int *launches, bool profiled = true);
// The top-K of score rows on the kernel csa2_set_topk_kernel chose (0 auto,
// 1 cluster, 2 one CTA per row: cudaErrorInvalidValue when a row does not fit).
void set_topk_choice(int which);
cudaError_t launch_topk(const TopkRows &r, cudaStream_t stream, int *launches, bool profiled = true);
// True when launch_topk(r) runs the cluster kernel (the one that takes a
// sweep's histogram).
bool topk_runs_cluster(const TopkRows &r);

// Chunked prefill: multi-query indexer over the causally visible entries.
struct PrefillIdxArgs {
  const float *w;             // [B*T][32] head weights of every chunk token
  float *scores;              // [groups*8][row_len] (block-local query rows)
  int64_t cap;                // entries per sequence in the caches
  int64_t row_len;            // tiles * 128
  int64_t first_pos;          // position of chunk token 0
  int64_t tokens;             // chunk tokens per sequence (multiple of 8)
  int64_t q0;                 // first flattened query token (b*tokens + i) of this block
  int64_t groups;             // groups of 8 tokens in this block
  int32_t ranges;             // key-tile ranges per group
  int32_t range_tiles;        // tiles per range
  int32_t tiles;              // key tiles every group covers (block maximum)
  int32_t m;                  // compression ratio
};

cudaError_t launch_prefill_indexer(const CUtensorMap &tm_k, const CUtensorMap &tm_q, const PrefillIdxArgs &a,
                                   int num_sms, cudaStream_t stream, int *launches);

size_t topk_scratch_bytes(int32_t rows, int64_t row_len, int32_t k);
TopkScratch carve_topk_scratch(void *base, int32_t rows, int64_t row_len, int32_t k);
// The HSI pool selection: for k <= 2048 the cluster top-K over a copy of the
// rows with the forced block set to +inf (in `scratch`, which must hold
// topk_scratch_bytes(rows, row_len, k)); the multi-pass top-K above that.
cudaError_t launch_pool_topk(const TopkRows &r, void *scratch, int num_sms, cudaStream_t stream, int *launches);
cudaError_t launch_topk(const TopkRows &r, const TopkScratch &s, int num_sms, cudaStream_t stream, int *launches);

struct AttnArgs {
  const __nv_bfloat16 *q;     // [P][64][512]
  const uint8_t *kv;          // [B][cap][288]
  const int32_t *idx;         // [P][K]
  const uint8_t *swa;         // [P][W][512] (E4M3)
  const float *swa_scale;     // [P][W]
  const int32_t *swa_len;     // [P]
  float *out;                 // [P][64][512]
  float *lse;                 // [P][64] or NULL
  int64_t cap;
  int32_t problems;
  int32_t K;
  int32_t W;
  int32_t C;                  // chunks per token (1, 2, 4, 8): the CTAs of one cluster when > 1
  int32_t Bk;                 // rows per key block (<= 128, or <= 160 with one block per CTA)
  // Problem p of this launch is token gp = p0 + p; it reads the caches of
  // sequence gp / tokens.  Decode: tokens = 1, SWA rows [gp*W, gp*W + swa_len[gp]).
  // Prefill (causal_swa): token i of its sequence sits at position
  // first_pos + i and reads the SWA rows of positions max(pos - W + 1, 0) .. pos,
  // row r of a sequence holding position swa_first_pos + r.
  int64_t p0;
  int64_t tokens;
  int32_t causal_swa;
  int64_t first_pos;
  int64_t swa_first_pos;
  int64_t swa_seq_rows;
  int32_t kernel;             // 0 automatic, 1 split into chunks, 2 one chunk per token
};

// Workspace of one readout launch (the chunk partials when tokens are split).
size_t attn_scratch_bytes(int32_t problems, int32_t K, int32_t W, int32_t kernel);
// Reads and clears the readout's own device error word (that unit is
// compiled as whole-program device code).
cudaError_t attn_take_error(unsigned int *bits);
cudaError_t launch_sparse_attn(AttnArgs a, void *scratch, cudaStream_t stream, int *launches);

}  // namespace csa2
