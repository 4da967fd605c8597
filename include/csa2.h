/*
 * csa2.h -- C ABI of the CSA2 sparse FP4 decode library (libcsa2.so, sm_103a).
 *
 * The calls follow the pages' statement of the decode-time CSA2 global
 * attention of DeepSeek-V4.1-Flash:
 *   [A] "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression"
 *       (en.mycoding.id): 2.3.1 the compressor and the projected Indexer K,
 *       2.3.2 cross-layer KV/index reuse, 2.3.3 the encoder's groups, 2.3.4
 *       Hierarchical Sparse Indexer, 2.4.4 FP4 Main KV Cache and FP4 indexer
 *       Q/K, 3.1 entry sizes, 3.3.1-3.3.3 sparse readout and the
 *       Full/Reindex/Reuse modes.
 *   [N] "DeepSeek-V4.1-Flash - Architecture" (notes.nimendra.online):
 *       section 2 (CSA2 modes table, layer schedule, main attention settings),
 *       section 3 (Hierarchical Sparse Indexer), section 4 (KV cache formats).
 *
 * Calls: csa2_kv_quant_write (new main-KV entries), csa2_kv_quant_write_ik
 * (the same plus each entry's projected indexer key), csa2_indexer_k_quant
 * (MXFP4 indexer-K entries), csa2_indexer_score_topk (indexer + top-K, Full
 * or Reindex), csa2_hier_pool_select (+ _static: the HSI pool),
 * csa2_sparse_attn (the readout), csa2_sparse_decode (one layer in a mode),
 * csa2_prefill_chunk (a chunk at m = 2); helpers csa2_workspace_bytes,
 * csa2_get_device_status, csa2_status_string, csa2_default_params,
 * csa2_entry_bytes, csa2_indexer_entry_bytes, csa2_last_launch_count,
 * csa2_set_profile_events, csa2_set_topk_kernel.
 *
 * Conventions for every call:
 *  - All tensor pointers are DEVICE pointers, caller-owned; the library never
 *    allocates or frees memory.  Between calls it keeps only a per-device
 *    error word (see csa2_get_device_status), the per-thread launch count of
 *    the last call (csa2_last_launch_count), the process-wide top-K kernel
 *    choice (csa2_set_topk_kernel) and, on each device that has run
 *    csa2_hier_pool_select_static, that call's static scratch array, which
 *    holds the last call's contents.
 *  - Every call is asynchronous on `stream` (NULL = legacy default stream) and
 *    returns CSA2_OK once its kernels are enqueued.  Host-side validation
 *    failures return an error code without launching anything.
 *  - bf16 tensors are passed as `const void*` (IEEE bfloat16, row-major).
 *  - Shapes are fixed by [N] section 2: latent / query head dim D = 512 with
 *    the last 64 channels RoPE'd, H = 64 query heads, 32 indexer heads of 128
 *    dims.  index_topk, sliding_window, candidate_block_size and
 *    candidate_topk_blocks come from csa2_params.
 *  - Pointers that kernels read with 16-byte vectors or TMA must be 16-byte
 *    aligned (noted per argument); a misaligned pointer is rejected.
 *  - Device-side checks (n_vis out of range, an index outside the cache, a
 *    bounded wait that ran out) never trap: they set bits in the device error
 *    word, which csa2_get_device_status reads and clears.
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *csa2_stream_t; /* the same type as cudaStream_t */

typedef enum {
  CSA2_OK = 0,
  CSA2_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, bad size or mode */
  CSA2_ERR_UNSUPPORTED = 2,  /* parameter outside the supported range       */
  CSA2_ERR_WORKSPACE = 3,    /* ws_bytes below csa2_workspace_bytes(...)    */
  CSA2_ERR_CUDA = 4,         /* a CUDA runtime call or launch failed         */
  CSA2_ERR_DEVICE = 5        /* device-detected fault, see the error bits    */
} csa2_status;

/* Device error bits returned through csa2_get_device_status(). */
#define CSA2_DEV_ERR_NVIS     0x1u  /* n_vis[b] < 0 or > n_max                 */
#define CSA2_DEV_ERR_INDEX    0x2u  /* an index / slot outside the cache        */
#define CSA2_DEV_ERR_TIMEOUT  0x4u  /* a bounded mbarrier wait ran out          */
#define CSA2_DEV_ERR_POOL     0x8u  /* a pool block id out of range / unsorted  */

/* The three CSA2 modes ([N] section 2 "CSA2 modes" table):
 *   FULL    new top-K from a sweep over all visible positions (and, with
 *           params.hsi, the HSI candidate pool), then the sparse readout;
 *   REINDEX reuse the cache, new top-K scored only over the candidate pool;
 *   REUSE   reuse the latest top-K, readout only. */
typedef enum { CSA2_MODE_FULL = 0, CSA2_MODE_REINDEX = 1, CSA2_MODE_REUSE = 2 } csa2_mode;

typedef struct {
  int32_t index_topk;            /* K, 1..2048; pages: 512                      */
  int32_t sliding_window;        /* W rows of SWA per query, 0..1024; pages: 128 */
  int32_t candidate_block_size;  /* HSI block width; must be 8 ([A] 2.3.4)      */
  int32_t candidate_topk_blocks; /* HSI pool blocks, 16..8192, multiple of 16; 2048 */
  int32_t block_reduce;          /* 0 = max over the block (pages), 1 = sum      */
  int32_t hsi;                   /* FULL: also build the candidate pool (1/0)    */
  int32_t attn_kernel;           /* readout work split: 0 automatic, 1 a token's
                                    keys split over a cluster of CTAs (at
                                    least 2 chunks), 2 one CTA per token (its
                                    keys in blocks of 128); the result is the
                                    same up to rounding                        */
  int32_t indexer_fp4;           /* 0: indexer K cache bf16 [.][128]; 1: MXFP4
                                    (csa2_indexer_k_quant) and the indexer
                                    query quantised to MXFP4 as well ([A] 2.4.4:
                                    "FP4 Indexer Q and K"; [A] 3.1: 68 B per
                                    entry).  Decode only.                      */
} csa2_params;

/* Defaults of the pages: K=512, W=128, blocks of 8, 2048 blocks, max, hsi=1. */
csa2_params csa2_default_params(void);

/* Bytes of one FP4 main-KV entry: 256 B of E2M1 codes (channel 2j in the low
 * nibble of byte j, 2j+1 in the high nibble) followed by 32 one-byte E4M3
 * scales (scale g covers channels 16g..16g+15).  = 288. */
int32_t csa2_entry_bytes(void);

/* Bytes of one indexer-K entry: 256 (bf16, 128 dims) or, with fp4 != 0, 68
 * (MXFP4: 64 B of E2M1 codes and 4 UE8M0 scale bytes, [A] 3.1). */
int32_t csa2_indexer_entry_bytes(int32_t fp4);

/*
 * csa2_kv_quant_write -- write new main-KV entries ([A] 2.4.4 "quantized after
 * RoPE"; [N] section 4; the compressor of [A] 2.3.1 at m = 2).
 *   For entry i: e = latent[i] (m = 1), or the channel-wise softmax-weighted
 *   pool of its m = 2 source latents with logits z[i] (computed in double,
 *   rounded once to fp32); RoPE on channels 448..511 as interleaved pairs at
 *   position entry_pos[i] with inverse frequency fl32(rope_theta^(-2j/64));
 *   then per 16 channels scale = E4M3_rne_satfinite(amax / 6) and codes =
 *   E2M1_rne_satfinite(x / scale) (all-zero codes when the scale is zero).
 *   latent    bf16 [n_entries][m][512], 16-byte aligned
 *   z         bf16 [n_entries][m][512] for m = 2, NULL for m = 1
 *   m         1 or 2
 *   entry_pos int64 [n_entries] RoPE positions
 *   slot      int64 [n_entries] destination row in kv, 0 <= slot < kv_rows
 *             (an out-of-range slot is skipped and sets CSA2_DEV_ERR_INDEX)
 *   kv        uint8 [kv_rows][288], 16-byte aligned
 * n_entries == 0 is a no-op.
 */
csa2_status csa2_kv_quant_write(const void *latent, const void *z, int32_t m, int64_t n_entries,
                                const int64_t *entry_pos, const int64_t *slot, uint8_t *kv,
                                int64_t kv_rows, float rope_theta, csa2_stream_t stream);

/*
 * csa2_kv_quant_write_ik -- csa2_kv_quant_write that also writes each
 * entry's indexer key, the Full layer's projection of its main-KV entry
 * ([A] 2.3.1: "obtains the Indexer K by projecting the main KV entries").
 *   k = W_ik e, e the entry before FP4 quantisation (compressed at m = 2,
 *   RoPE'd, fp32), fp32 accumulation, rounded to bf16 (nearest even); with
 *   indexer_fp4 the bf16 row is then written as MXFP4 exactly as
 *   csa2_indexer_k_quant writes it.
 *   w_ik   bf16 [128][512] (row-major), 16-byte aligned
 *   k_idx  bf16 [k_rows][128], or with indexer_fp4 the MXFP4 planes of k_rows
 *          rows (k_rows a multiple of 4); 16-byte aligned
 *   row slot[i] of both caches is written; slot[i] >= k_rows is skipped and
 *   sets CSA2_DEV_ERR_INDEX.  Other arguments as csa2_kv_quant_write.
 */
csa2_status csa2_kv_quant_write_ik(const void *latent, const void *z, int32_t m, int64_t n_entries,
                                   const int64_t *entry_pos, const int64_t *slot, uint8_t *kv, int64_t kv_rows,
                                   float rope_theta, const void *w_ik, void *k_idx, int64_t k_rows,
                                   int32_t indexer_fp4, csa2_stream_t stream);

/*
 * csa2_indexer_k_quant -- write MXFP4 indexer-K entries (OCP Microscaling:
 * blocks of 32 dims share one UE8M0 scale 2^E, E = floor(log2(max |x|)) - 2
 * clamped to [-127, 127] (-127 for an all-zero block); codes =
 * E2M1_rne_satfinite(x / 2^E)).  The cache holds two planes: codes
 * [rows][64] (dim 2j in the low nibble of byte j) at k_fp4, then scales
 * [rows][4] (byte E + 127 for dims 32i..32i+31) at k_fp4 + rows * 64: 68 B per
 * entry ([A] 3.1).
 *   k      bf16 [n][128], 16-byte aligned
 *   slot   int64 [n] destination rows, 0 <= slot < rows (others are skipped
 *          and set CSA2_DEV_ERR_INDEX)
 *   k_fp4  uint8 [rows * 68], 16-byte aligned; rows a multiple of 4
 * n == 0 is a no-op.
 */
csa2_status csa2_indexer_k_quant(const void *k, int64_t n, const int64_t *slot, uint8_t *k_fp4, int64_t rows,
                                 csa2_stream_t stream);

/*
 * csa2_indexer_score_topk -- lightning indexer + top-K ([N] sections 2-3,
 * [A] 2.3.4).  For sequence b: score(n) = sum_h w[b][h] * ReLU(q_idx[b][h] .
 * k_idx[b][n]) in fp32 over 32 heads x 128 dims (bf16 tensor-core products,
 * fp32 accumulation), for
 *   pool_blocks == NULL (Full): every visible position n < n_vis[b];
 *   pool_blocks != NULL (Reindex): only the positions of the pool's blocks,
 *     pool_blocks[b][j]*8 + i for i < 8, truncated to n_vis[b].
 * topk_idx[b] receives the index_topk highest-scoring positions (ties toward
 * the lower position), ascending, -1 padded when fewer are visible.
 *   q_idx  bf16 [batch][32][128], 16-byte aligned
 *   w      fp32 [batch][32]
 *   k_idx  bf16 [batch][cap][128], 16-byte aligned (indexer K cache); with
 *          params.indexer_fp4 the MXFP4 planes of csa2_indexer_k_quant with
 *          rows = batch * cap (cap a multiple of 4), and q_idx is quantised to
 *          MXFP4 the same way; the products are those of the dequantised
 *          values, taken on fp16 tensor cores as code x 2^(E - Emax) with
 *          2^Emax (the row's largest block scale) applied in fp32 after the
 *          dot product: exact for every block within 2^23 of its row's largest
 *   n_vis  int32 [batch], 0 <= n_vis[b] <= n_max <= cap (checked on device)
 *   n_max  host-side bound on n_vis, sizes the launch and the workspace
 *   pool_blocks int32 [batch][candidate_topk_blocks] ascending, -1 padded
 *   topk_idx    int32 [batch][index_topk] (out)
 *   block_scores fp32 [batch][ceil(n_max/8)] (out, Full only, may be NULL):
 *     per block of 8 positions the max (or sum) of its visible scores, -inf
 *     for blocks with no visible position -- the HSI block scores.
 *   ws / ws_bytes: scratch of at least csa2_workspace_bytes(...) bytes,
 *     256-byte aligned.  Its contents never change a result.  The bf16 sweep
 *     counts each row's scores by key range at the start of the workspace
 *     for the top-K, which then needs no sample of the row, and the top-K
 *     leaves those counts zero; a workspace that starts zeroed (or was last
 *     used by this entry point with the same batch and n_max) gives the
 *     first call that benefit too, any other contents only make that call's
 *     selection take a slower path.  csa2_sparse_decode keeps the same counts
 *     in its own workspace, in a place its other steps leave untouched.
 */
csa2_status csa2_indexer_score_topk(const void *q_idx, const float *w, const void *k_idx,
                                    int32_t batch, int64_t cap, const int32_t *n_vis,
                                    int64_t n_max, const int32_t *pool_blocks,
                                    const csa2_params *params, int32_t *topk_idx,
                                    float *block_scores, void *ws, size_t ws_bytes,
                                    csa2_stream_t stream);

/*
 * csa2_hier_pool_select -- the HSI candidate pool ([A] 2.3.4, [N] section 3).
 * From the block scores of a Full layer: the block holding position
 * n_vis[b]-1 is forced in (its score taken as +inf), then the
 * candidate_topk_blocks highest blocks (ties toward the lower block) are kept.
 *   block_scores fp32 [batch][ceil(n_max/8)] as written by
 *     csa2_indexer_score_topk (-inf marks blocks past n_vis)
 *   pool_blocks  int32 [batch][candidate_topk_blocks] (out) ascending, -1 padded
 */
csa2_status csa2_hier_pool_select(const float *block_scores, const int32_t *n_vis,
                                  int32_t batch, int64_t n_max, const csa2_params *params,
                                  int32_t *pool_blocks, void *ws, size_t ws_bytes,
                                  csa2_stream_t stream);

/*
 * csa2_sparse_attn -- the sparse readout alone ([A] 3.3.1-3.3.2, [N] section 2).
 * For each sequence b and head h: one softmax over the selected main-KV
 * entries {kv[b][topk_idx[b][j]] : topk_idx >= 0} together with the SWA rows
 * {swa[b][t] : t < swa_len[b]}, logits q . k / sqrt(512); key = value = the
 * dequantised 512-d latent (FP4 code x E4M3 scale, resp. E4M3 x the row's fp32
 * scale).  out = the convex combination; lse = natural log of the softmax
 * denominator (-inf, with out = 0, when there is no key).
 *   q         bf16 [batch][64][512], 16-byte aligned (|q| below 65504)
 *   kv        uint8 [batch][cap][288], 16-byte aligned
 *   topk_idx  int32 [batch][index_topk], entries in [-1, cap)
 *   swa       uint8 E4M3 [batch][sliding_window][512], 16-byte aligned
 *   swa_scale fp32 [batch][sliding_window]
 *   swa_len   int32 [batch], 0..sliding_window
 *   out       fp32 [batch][64][512] (out); lse fp32 [batch][64] or NULL (out)
 */
csa2_status csa2_sparse_attn(const csa2_params *params, int32_t batch, const void *q,
                             const uint8_t *kv, int64_t cap, const int32_t *topk_idx,
                             const uint8_t *swa, const float *swa_scale, const int32_t *swa_len,
                             float *out, float *lse, void *ws, size_t ws_bytes,
                             csa2_stream_t stream);

/*
 * csa2_sparse_decode -- one CSA2 layer of a decode step, by mode ([N]
 * section 2 modes table and layer schedule; [A] 3.3.3):
 *   FULL    csa2_indexer_score_topk over all visible positions -> topk_idx (out);
 *           with params.hsi also csa2_hier_pool_select -> pool_blocks (out);
 *           then csa2_sparse_attn.
 *   REINDEX csa2_indexer_score_topk over pool_blocks (in) -> topk_idx (out);
 *           then csa2_sparse_attn.
 *   REUSE   csa2_sparse_attn with topk_idx (in) from the latest index layer;
 *           q_idx, w, k_idx and pool_blocks are not read (may be NULL).
 * Writing the new token's main-KV entry (csa2_kv_quant_write) is a separate
 * call the caller makes before the Full layer.  Arguments as above.
 */
csa2_status csa2_sparse_decode(csa2_mode mode, const csa2_params *params, int32_t batch,
                               const void *q, const void *q_idx, const float *w,
                               const uint8_t *kv, const void *k_idx, int64_t cap,
                               const int32_t *n_vis, int64_t n_max, const uint8_t *swa,
                               const float *swa_scale, const int32_t *swa_len,
                               int32_t *topk_idx, int32_t *pool_blocks, float *out, float *lse,
                               void *ws, size_t ws_bytes, csa2_stream_t stream);

/*
 * csa2_prefill_chunk -- the indexer, top-K and sparse readout of every token
 * of a prefill chunk ([N] section 1-2: the encoder's CSA2 layers at m = 2;
 * [A] 2.3.1-2.3.3).  Token i (0 <= i < n_tokens) of sequence b sits at position
 * pos = first_pos + i and sees the compressed entries j with m*j + m-1 <= pos
 * (an entry is visible once all its m source tokens are).  For each token:
 * score(j) = sum_h w_h ReLU(q_idx_h . k_j) over its visible entries (bf16
 * tensor-core products, fp32), the index_topk best (ties toward the lower
 * entry, ascending, -1 padded), then one softmax over those entries together
 * with the token's own causal SWA window -- the rows of positions
 * max(pos - sliding_window + 1, 0) .. pos -- as in csa2_sparse_attn.  The
 * chunk's own entries must already be in the caches (csa2_kv_quant_write with
 * m = 2 for the chunk's complete pairs).
 *   q         bf16 [batch][n_tokens][64][512], 16-byte aligned
 *   q_idx     bf16 [batch][n_tokens][32][128], 16-byte aligned
 *   w         fp32 [batch][n_tokens][32], 16-byte aligned
 *   kv        uint8 [batch][cap][288]; k_idx bf16 [batch][cap][128]
 *   n_tokens  a multiple of 8; (first_pos + n_tokens) / m <= cap
 *   m         1 or 2
 *   swa       uint8 E4M3 [batch][swa_rows][512]; swa_scale fp32 [batch][swa_rows];
 *             row r of a sequence holds position swa_first_pos + r, and must
 *             cover every window (swa_first_pos <= max(first_pos - W + 1, 0),
 *             first_pos + n_tokens - 1 < swa_first_pos + swa_rows)
 *   topk_idx  int32 [batch][n_tokens][index_topk] (out)
 *   out       fp32 [batch][n_tokens][64][512] (out); lse fp32 [batch][n_tokens][64] or NULL
 *   ws        at least csa2_workspace_bytes(CSA2_OP_PREFILL, batch, cap, params)
 * The chunk is processed in blocks of 1024 tokens (indexer, top-K, readout per block).
 */
csa2_status csa2_prefill_chunk(const csa2_params *params, int32_t batch, int32_t n_tokens, int64_t first_pos,
                               int32_t m, const void *q, const void *q_idx, const float *w,
                               const uint8_t *kv, const void *k_idx, int64_t cap, const uint8_t *swa,
                               const float *swa_scale, int64_t swa_rows, int64_t swa_first_pos,
                               int32_t *topk_idx, float *out, float *lse, void *ws, size_t ws_bytes,
                               csa2_stream_t stream);

/*
 * csa2_hier_pool_select_static -- csa2_hier_pool_select without a workspace.
 * The pages have no counterpart to this call; it exists for callers that
 * cannot allocate device memory where they select the pool: a runtime that
 * replays a fixed, pre-planned memory layout and forbids allocation while it
 * executes, or host code that holds only raw pointers to its inputs and
 * outputs and has no allocator to ask for scratch.
 * Same arguments and result as csa2_hier_pool_select, minus ws / ws_bytes.
 * The scratch is a static device array of CSA2_POOL_STATIC_SCRATCH_BYTES
 * (16 MiB) inside this library, held by every GPU that loads it until the
 * process exits.  The call never allocates or frees memory.  Its first call on
 * a device looks up that array's device address (once per device, with the
 * device current), so make that first call before any stream capture.  A
 * request needing more scratch than the array holds (about batch *
 * ceil(n_max/8) * 8 bytes of candidates plus 8 KB and 4 * candidate_topk_blocks
 * bytes per sequence) returns CSA2_ERR_WORKSPACE without launching.  All calls
 * on a device share the array and it keeps the last call's contents; each call
 * clears the counters it needs first, and calls that overlap on the GPU
 * (other streams or host threads) race on it and must be serialised by the
 * caller.
 */
#define CSA2_POOL_STATIC_SCRATCH_BYTES ((size_t)16 << 20)
csa2_status csa2_hier_pool_select_static(const float *block_scores, const int32_t *n_vis,
                                         int32_t batch, int64_t n_max, const csa2_params *params,
                                         int32_t *pool_blocks, csa2_stream_t stream);

/* Operation selector for csa2_workspace_bytes. */
typedef enum {
  CSA2_OP_INDEXER = 0,   /* csa2_indexer_score_topk        */
  CSA2_OP_POOL = 1,      /* csa2_hier_pool_select          */
  CSA2_OP_ATTN = 2,      /* csa2_sparse_attn               */
  CSA2_OP_DECODE = 3,    /* csa2_sparse_decode (any mode)  */
  CSA2_OP_PREFILL = 4    /* csa2_prefill_chunk (n_max = cap) */
} csa2_op;

/* Scratch bytes an operation needs for `batch` sequences and visible
 * lengths up to n_max.  0 on invalid arguments. */
size_t csa2_workspace_bytes(csa2_op op, int32_t batch, int64_t n_max, const csa2_params *params);

/* Synchronises `stream`, then returns and clears the current device's error
 * word (CSA2_DEV_ERR_* bits, 0 if none) in *bits (may be NULL).  Returns
 * CSA2_ERR_DEVICE if any bit was set, CSA2_ERR_CUDA if the synchronisation
 * failed, else CSA2_OK. */
csa2_status csa2_get_device_status(csa2_stream_t stream, uint32_t *bits);

/* Static text for a status code. */
const char *csa2_status_string(csa2_status s);

/* Number of kernels the last successful call on this thread enqueued. */
int32_t csa2_last_launch_count(void);

/* Timing hook for benchmarks: when `start` and `stop` (cudaEvent_t handles)
 * are non-NULL, later calls on this thread record `start` on their stream
 * right before every launch of the chosen kernel and `stop` right after it
 * (kernel 0 = the indexer sweep, 1 = the sparse-attention kernel, 2 = the
 * chunked-prefill indexer, 3 = the top-K selection).  NULL
 * handles switch the hook off.  Events recorded during stream capture become
 * part of the captured graph. */
typedef enum {
  CSA2_KERNEL_INDEXER_SWEEP = 0,
  CSA2_KERNEL_SPARSE_ATTN = 1,
  CSA2_KERNEL_PREFILL_INDEXER = 2,
  CSA2_KERNEL_TOPK = 3
} csa2_kernel;
csa2_status csa2_set_profile_events(csa2_kernel kernel, void *start, void *stop);

/* Which kernel the top-K selections (index_topk of the Full and Reindex
 * layers and of prefill, the HSI pool) run on, for tests and measurements:
 * 0 = automatic (one CTA per row for rows of at most 131,072 scores when a
 * call has at least twice as many rows as the GPU has SMs, else one
 * thread-block cluster per row), 1 = one
 * cluster per row, 2 = one CTA per row (a call whose rows do not fit then
 * fails with CSA2_ERR_CUDA).  Both kernels are exact and give the same
 * result.  Applies to later calls in this process;
 * CSA2_ERR_INVALID_ARG for any other value. */
csa2_status csa2_set_topk_kernel(int32_t which);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
