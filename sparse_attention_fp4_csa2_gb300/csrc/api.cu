// C ABI of the CSA2 library: argument checks, workspace layout, TMA tensor
// maps and the launch sequence of each call (declared in include/csa2.h).
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "kernels.cuh"

namespace csa2 {

__device__ unsigned int g_dev_error = 0;

namespace {
thread_local ProfileEvents g_profile[4];
}

ProfileEvents &profile_events(int kernel) { return g_profile[kernel >= 0 && kernel < 4 ? kernel : 0]; }

namespace {
thread_local int32_t g_last_launches = 0;
}

void set_last_launch_count(int32_t n) { g_last_launches = n; }

cudaError_t record_profile_event(cudaEvent_t ev, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cs);
  if (e != cudaSuccess) return e;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, stream);
}

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

int num_sms() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 1;
  return n;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

}  // namespace

// 2-D bf16 tensor map over rows of `inner` elements, box {64, box_rows}, 128B swizzle.
bool make_tmap_bf16(CUtensorMap *m, const void *ptr, int64_t inner, int64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)inner * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

bool make_tmap_bf16_rows128(CUtensorMap *m, const void *ptr, int64_t rows, uint32_t box_rows) {
  return make_tmap_bf16(m, ptr, 128, rows, box_rows);
}

// 2-D byte tensor map over rows of 64 B, box {64, box_rows}, 64B swizzle.
bool make_tmap_u8_rows64(CUtensorMap *m, const void *ptr, int64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {64, (cuuint64_t)rows};
  cuuint64_t strides[1] = {64};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D byte tensor map over rows of 128 B, box {128, box_rows}, 128B swizzle.
bool make_tmap_u8_rows128(CUtensorMap *m, const void *ptr, int64_t rows, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {128, (cuuint64_t)rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool params_ok(const csa2_params *p) {
  return p && p->index_topk >= 1 && p->index_topk <= 2048 && p->sliding_window >= 0 &&
         p->sliding_window <= 1024 && p->candidate_block_size == BLOCK && p->candidate_topk_blocks >= 16 &&
         p->candidate_topk_blocks <= TOPK_MAX_K && p->candidate_topk_blocks % 16 == 0 &&
         (p->block_reduce == 0 || p->block_reduce == 1) && (p->hsi == 0 || p->hsi == 1) &&
         p->attn_kernel >= 0 && p->attn_kernel <= 2 && (p->indexer_fp4 == 0 || p->indexer_fp4 == 1);
}

// ------------------------------------------------------------ workspace
// The rows' score histograms, handed from the sweep to the top-K: at the
// start of the indexer's workspace, in the same place for Full and Reindex
// calls, and kept out of the pool selection's and the readout's scratch in a
// decode call (the top-K leaves them zero for the next call).
size_t hist_ws(int32_t batch) { return (size_t)round_up((int64_t)batch * TOPK_HIST_BINS * 4, 256); }

struct IndexerLayout {
  int64_t row_len;       // scores per row
  size_t hist_off, scores_off, q8_off, wq_off, end;
};

IndexerLayout indexer_layout(int32_t batch, int64_t n_max, const csa2_params *p, bool pool) {
  IndexerLayout L;
  const bool fp4 = p->indexer_fp4 != 0;
  L.row_len = pool ? (int64_t)p->candidate_topk_blocks * BLOCK : round_up(n_max, fp4 ? FP4_SWEEP_TILE : SWEEP_TILE);
  L.hist_off = 0;
  L.scores_off = hist_ws(batch);
  L.q8_off = L.scores_off + (size_t)round_up((int64_t)batch * L.row_len * 4, 256);
  // MXFP4 indexer: the queries' E5M2 rows and the head weights with their
  // row exponents folded in; the cluster top-K needs no scratch beyond the scores
  L.wq_off = L.q8_off + (fp4 ? (size_t)round_up((int64_t)batch * HI * DI, 256) : 0);
  L.end = L.wq_off + (fp4 ? (size_t)round_up((int64_t)batch * HI * 4, 256) : 0);
  return L;
}

size_t indexer_ws(int32_t batch, int64_t n_max, const csa2_params *p) {
  const size_t a = indexer_layout(batch, n_max, p, false).end;
  const size_t b = indexer_layout(batch, n_max, p, true).end;
  return a > b ? a : b;
}

size_t pool_ws(int32_t batch, int64_t n_max, const csa2_params *p) {
  const int64_t nblk = (n_max + BLOCK - 1) / BLOCK;
  return topk_scratch_bytes(batch, nblk, p->candidate_topk_blocks);
}

size_t attn_ws(int32_t batch, const csa2_params *p) {
  return attn_scratch_bytes(batch, p->index_topk, p->sliding_window, p->attn_kernel);
}

size_t decode_ws(int32_t batch, int64_t n_max, const csa2_params *p) {
  const int64_t nblk = (n_max + BLOCK - 1) / BLOCK;
  size_t bs = (size_t)round_up((int64_t)batch * nblk * 4, 256);
  const size_t h = hist_ws(batch);
  size_t a = indexer_ws(batch, n_max, p) - h, b = pool_ws(batch, n_max, p), c = attn_ws(batch, p);
  size_t m = a > b ? a : b;
  m = m > c ? m : c;
  return bs + h + m;
}

constexpr int64_t kPrefillBlock = 1024;   // query tokens per indexer / top-K / attention block

size_t prefill_ws(int32_t batch, int64_t cap, const csa2_params *p) {
  const int64_t qb = kPrefillBlock;
  size_t b = (size_t)round_up(qb * round_up(cap, SWEEP_TILE) * 4, 256);
  b += attn_scratch_bytes((int32_t)qb, p->index_topk, p->sliding_window, p->attn_kernel);
  (void)batch;
  return b;
}

csa2_status cuda_status(cudaError_t e) { return e == cudaSuccess ? CSA2_OK : CSA2_ERR_CUDA; }

// ----------------------------------------------------------- operations
csa2_status run_indexer(const void *q_idx, const float *w, const void *k_idx, int32_t batch, int64_t cap,
                        const int32_t *n_vis, int64_t n_max, const int32_t *pool_blocks, const csa2_params *p,
                        int32_t *topk_idx, float *block_scores, void *ws, size_t ws_bytes, cudaStream_t stream,
                        int *launches) {
  if (!q_idx || !w || !k_idx || !n_vis || !topk_idx || !ws) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(q_idx) || !aligned16(k_idx) || (reinterpret_cast<uintptr_t>(ws) & 255u)) return CSA2_ERR_INVALID_ARG;
  if (batch < 1 || cap < 1 || n_max < 0 || n_max > cap) return CSA2_ERR_INVALID_ARG;
  if ((int64_t)batch * cap >= (int64_t)1 << 31 || (int64_t)batch * HI >= (int64_t)1 << 31) return CSA2_ERR_UNSUPPORTED;
  if (pool_blocks && block_scores) return CSA2_ERR_INVALID_ARG;
  if (ws_bytes < indexer_ws(batch, n_max, p)) return CSA2_ERR_WORKSPACE;
  const bool pool = pool_blocks != nullptr;
  const IndexerLayout L = indexer_layout(batch, n_max, p, pool);
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  float *scores = reinterpret_cast<float *>(wsb + L.scores_off);

  const bool fp4 = p->indexer_fp4 != 0;
  if (fp4 && cap % 4 != 0) return CSA2_ERR_INVALID_ARG;
  CUtensorMap tm_k, tm_q;
  float *wq = nullptr;
  if (fp4) {
    // the queries in MXFP4 (as E5M2 bytes), then the sweep over the planes
    void *q8 = wsb + L.q8_off;
    wq = reinterpret_cast<float *>(wsb + L.wq_off);
    if (launch_indexer_q_fp4(q_idx, w, (int64_t)batch * HI, q8, wq, stream) != cudaSuccess) return CSA2_ERR_CUDA;
    ++*launches;
    if (!make_tmap_u8_rows128(&tm_q, q8, (int64_t)batch * HI, HI)) return CSA2_ERR_CUDA;
    if (!make_tmap_u8_rows64(&tm_k, k_idx, (int64_t)batch * cap, pool ? BLOCK : FP4_SWEEP_TILE)) return CSA2_ERR_CUDA;
  } else {
    if (!make_tmap_bf16_rows128(&tm_k, k_idx, (int64_t)batch * cap, pool ? BLOCK : SWEEP_TILE)) return CSA2_ERR_CUDA;
    if (!make_tmap_bf16_rows128(&tm_q, q_idx, (int64_t)batch * HI, HI)) return CSA2_ERR_CUDA;
  }
  SweepArgs a;
  a.w = fp4 ? wq : w;
  a.n_vis = n_vis;
  a.pool = pool_blocks;
  a.scores = scores;
  a.block_scores = block_scores;
  a.cap = cap;
  a.n_max = n_max;
  a.row_len = L.row_len;
  a.batch = batch;
  a.tiles_per_seq = fp4 ? (int32_t)((L.row_len + FP4_SWEEP_TILE - 1) / FP4_SWEEP_TILE)
                        : (int32_t)(L.row_len / SWEEP_TILE);
  a.pool_nb = p->candidate_topk_blocks;
  a.nblk_stride = (int32_t)((n_max + BLOCK - 1) / BLOCK);
  a.block_reduce = p->block_reduce;
  a.k_scales = fp4 ? static_cast<const uint8_t *>(k_idx) + (int64_t)batch * cap * (DI / 2) : nullptr;
  a.k_rows = (int64_t)batch * cap;
  TopkRows r;
  r.vals = scores;
  r.row_len = L.row_len;
  r.row_stride = L.row_len;
  r.rows = batch;
  r.k = p->index_topk;
  r.force_nvis = nullptr;
  r.force_block = BLOCK;
  r.n_max = n_max;
  r.pool = pool_blocks;
  r.pool_stride = p->candidate_topk_blocks;
  r.out = topk_idx;
  // the bf16 sweep counts the rows' keys for the cluster top-K, which then
  // needs no sample of the scores (and clears the counts).  The MXFP4 sweep
  // does not: its epilogue shares issue slots with the code conversion, and
  // counting there cost it more than the top-K saved.
  if (!fp4 && topk_cluster_supported(r) && topk_runs_cluster(r)) {
    r.hist = reinterpret_cast<uint32_t *>(wsb + L.hist_off);
    a.hist = r.hist;
  }
  const int sms = num_sms();
  cudaError_t e = fp4 ? launch_indexer_sweep_fp4(tm_k, tm_q, a, sms, stream, launches)
                      : launch_indexer_sweep(tm_k, tm_q, a, sms, stream, launches);
  if (e != cudaSuccess) return CSA2_ERR_CUDA;
  return cuda_status(launch_topk(r, stream, launches));
}

csa2_status run_pool(const float *block_scores, const int32_t *n_vis, int32_t batch, int64_t n_max,
                     const csa2_params *p, int32_t *pool_blocks, void *ws, size_t ws_bytes, cudaStream_t stream,
                     int *launches) {
  if (!block_scores || !n_vis || !pool_blocks || !ws) return CSA2_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(ws) & 255u)) return CSA2_ERR_INVALID_ARG;
  if (batch < 1 || n_max < 0) return CSA2_ERR_INVALID_ARG;
  if (ws_bytes < pool_ws(batch, n_max, p)) return CSA2_ERR_WORKSPACE;
  const int64_t nblk = (n_max + BLOCK - 1) / BLOCK;
  TopkRows r;
  r.vals = block_scores;
  r.row_len = nblk;
  r.row_stride = nblk;
  r.rows = batch;
  r.k = p->candidate_topk_blocks;
  r.force_nvis = n_vis;
  r.force_block = BLOCK;
  r.n_max = n_max;
  r.pool = nullptr;
  r.pool_stride = 0;
  r.out = pool_blocks;
  return cuda_status(launch_pool_topk(r, ws, num_sms(), stream, launches));
}

csa2_status run_attn(const csa2_params *p, int32_t batch, const void *q, const uint8_t *kv, int64_t cap,
                     const int32_t *topk_idx, const uint8_t *swa, const float *swa_scale, const int32_t *swa_len,
                     float *out, float *lse, void *ws, size_t ws_bytes, cudaStream_t stream, int *launches) {
  if (!q || !kv || !topk_idx || !out || !ws) return CSA2_ERR_INVALID_ARG;
  if (p->sliding_window > 0 && (!swa || !swa_scale || !swa_len)) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(kv) || (swa && !aligned16(swa)) || (reinterpret_cast<uintptr_t>(ws) & 255u))
    return CSA2_ERR_INVALID_ARG;
  if (batch < 1 || batch > 65535 || cap < 1) return CSA2_ERR_INVALID_ARG;
  if (ws_bytes < attn_ws(batch, p)) return CSA2_ERR_WORKSPACE;
  AttnArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = static_cast<const __nv_bfloat16 *>(q);
  a.kv = kv;
  a.idx = topk_idx;
  a.swa = swa;
  a.swa_scale = swa_scale;
  a.swa_len = swa_len;
  a.out = out;
  a.lse = lse;
  a.cap = cap;
  a.problems = batch;
  a.K = p->index_topk;
  a.W = p->sliding_window;
  a.p0 = 0;
  a.tokens = 1;
  a.causal_swa = 0;
  a.kernel = p->attn_kernel;
  return cuda_status(launch_sparse_attn(a, ws, stream, launches));
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" {

csa2_params csa2_default_params(void) {
  csa2_params p;
  p.index_topk = 512;
  p.sliding_window = 128;
  p.candidate_block_size = 8;
  p.candidate_topk_blocks = 2048;
  p.block_reduce = 0;
  p.hsi = 1;
  p.attn_kernel = 0;
  p.indexer_fp4 = 0;
  return p;
}

int32_t csa2_entry_bytes(void) { return ENTRY_BYTES; }

int32_t csa2_last_launch_count(void) { return g_last_launches; }

csa2_status csa2_set_profile_events(csa2_kernel kernel, void *start, void *stop) {
  if (kernel != CSA2_KERNEL_INDEXER_SWEEP && kernel != CSA2_KERNEL_SPARSE_ATTN &&
      kernel != CSA2_KERNEL_PREFILL_INDEXER && kernel != CSA2_KERNEL_TOPK)
    return CSA2_ERR_INVALID_ARG;
  ProfileEvents &pe = profile_events(kernel);
  pe.start = static_cast<cudaEvent_t>(start);
  pe.stop = static_cast<cudaEvent_t>(stop);
  return CSA2_OK;
}

csa2_status csa2_set_topk_kernel(int32_t which) {
  if (which < 0 || which > 2) return CSA2_ERR_INVALID_ARG;
  set_topk_choice(which);
  return CSA2_OK;
}

int32_t csa2_indexer_entry_bytes(int32_t fp4) { return fp4 ? DI / 2 + DI / 32 : DI * 2; }

const char *csa2_status_string(csa2_status s) {
  switch (s) {
    case CSA2_OK: return "ok";
    case CSA2_ERR_INVALID_ARG: return "invalid argument";
    case CSA2_ERR_UNSUPPORTED: return "unsupported parameter";
    case CSA2_ERR_WORKSPACE: return "workspace too small";
    case CSA2_ERR_CUDA: return "CUDA error";
    case CSA2_ERR_DEVICE: return "device-side error";
  }
  return "unknown status";
}

size_t csa2_workspace_bytes(csa2_op op, int32_t batch, int64_t n_max, const csa2_params *params) {
  if (!params_ok(params) || batch < 1 || n_max < 0) return 0;
  switch (op) {
    case CSA2_OP_INDEXER: return indexer_ws(batch, n_max, params);
    case CSA2_OP_POOL: return pool_ws(batch, n_max, params);
    case CSA2_OP_ATTN: return attn_ws(batch, params);
    case CSA2_OP_DECODE: return decode_ws(batch, n_max, params);
    case CSA2_OP_PREFILL: return prefill_ws(batch, n_max, params);
  }
  return 0;
}

csa2_status csa2_get_device_status(csa2_stream_t stream, uint32_t *bits) {
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return CSA2_ERR_CUDA;
  unsigned int v = 0, zero = 0, va = 0;
  if (cudaMemcpyFromSymbol(&v, g_dev_error, sizeof(v)) != cudaSuccess) return CSA2_ERR_CUDA;
  if (v && cudaMemcpyToSymbol(g_dev_error, &zero, sizeof(zero)) != cudaSuccess) return CSA2_ERR_CUDA;
  if (attn_take_error(&va) != cudaSuccess) return CSA2_ERR_CUDA;   // the readout's own word
  v |= va;
  if (bits) *bits = v;
  return v ? CSA2_ERR_DEVICE : CSA2_OK;
}

csa2_status csa2_kv_quant_write(const void *latent, const void *z, int32_t m, int64_t n_entries,
                                const int64_t *entry_pos, const int64_t *slot, uint8_t *kv, int64_t kv_rows,
                                float rope_theta, csa2_stream_t stream) {
  g_last_launches = 0;
  if (n_entries < 0 || kv_rows < 0 || (m != 1 && m != 2)) return CSA2_ERR_INVALID_ARG;
  if (n_entries == 0) return CSA2_OK;
  if (!latent || !entry_pos || !slot || !kv || (m == 2 && !z)) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(latent) || !aligned16(kv) || (z && !aligned16(z))) return CSA2_ERR_INVALID_ARG;
  if (!(rope_theta > 1.0f)) return CSA2_ERR_INVALID_ARG;
  if (n_entries > ((int64_t)1 << 34)) return CSA2_ERR_UNSUPPORTED;
  const cudaError_t e = launch_kv_quant_write(latent, m == 2 ? z : nullptr, m, n_entries, entry_pos, slot, kv,
                                              kv_rows, rope_theta, reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return CSA2_ERR_CUDA;
  g_last_launches = 1;
  return CSA2_OK;
}

csa2_status csa2_kv_quant_write_ik(const void *latent, const void *z, int32_t m, int64_t n_entries,
                                   const int64_t *entry_pos, const int64_t *slot, uint8_t *kv, int64_t kv_rows,
                                   float rope_theta, const void *w_ik, void *k_idx, int64_t k_rows, int32_t indexer_fp4,
                                   csa2_stream_t stream) {
  g_last_launches = 0;
  if (n_entries < 0 || kv_rows < 0 || k_rows < 0 || (m != 1 && m != 2) || (indexer_fp4 != 0 && indexer_fp4 != 1))
    return CSA2_ERR_INVALID_ARG;
  if (indexer_fp4 && k_rows % 4 != 0) return CSA2_ERR_INVALID_ARG;
  if (n_entries == 0) return CSA2_OK;
  if (!latent || !entry_pos || !slot || !kv || (m == 2 && !z) || !w_ik || !k_idx) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(latent) || !aligned16(kv) || (z && !aligned16(z)) || !aligned16(w_ik) || !aligned16(k_idx))
    return CSA2_ERR_INVALID_ARG;
  if (!(rope_theta > 1.0f)) return CSA2_ERR_INVALID_ARG;
  if (n_entries > ((int64_t)1 << 34)) return CSA2_ERR_UNSUPPORTED;
  const cudaError_t e =
      launch_kv_quant_write(latent, m == 2 ? z : nullptr, m, n_entries, entry_pos, slot, kv, kv_rows, rope_theta,
                            reinterpret_cast<cudaStream_t>(stream), w_ik, k_idx, k_rows, indexer_fp4);
  if (e != cudaSuccess) return CSA2_ERR_CUDA;
  g_last_launches = 1;
  return CSA2_OK;
}

csa2_status csa2_indexer_k_quant(const void *k, int64_t n, const int64_t *slot, uint8_t *k_fp4, int64_t rows,
                                 csa2_stream_t stream) {
  g_last_launches = 0;
  if (n < 0 || rows < 0 || rows % 4 != 0) return CSA2_ERR_INVALID_ARG;
  if (n == 0) return CSA2_OK;
  if (!k || !slot || !k_fp4 || !aligned16(k) || !aligned16(k_fp4)) return CSA2_ERR_INVALID_ARG;
  if (n > ((int64_t)1 << 34)) return CSA2_ERR_UNSUPPORTED;
  if (launch_indexer_k_quant(k, n, slot, k_fp4, rows, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return CSA2_ERR_CUDA;
  g_last_launches = 1;
  return CSA2_OK;
}

csa2_status csa2_indexer_score_topk(const void *q_idx, const float *w, const void *k_idx, int32_t batch, int64_t cap,
                                    const int32_t *n_vis, int64_t n_max, const int32_t *pool_blocks,
                                    const csa2_params *params, int32_t *topk_idx, float *block_scores, void *ws,
                                    size_t ws_bytes, csa2_stream_t stream) {
  g_last_launches = 0;
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  int launches = 0;
  const csa2_status s = run_indexer(q_idx, w, k_idx, batch, cap, n_vis, n_max, pool_blocks, params, topk_idx,
                                    block_scores, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), &launches);
  if (s == CSA2_OK) g_last_launches = launches;
  return s;
}

csa2_status csa2_hier_pool_select(const float *block_scores, const int32_t *n_vis, int32_t batch, int64_t n_max,
                                  const csa2_params *params, int32_t *pool_blocks, void *ws, size_t ws_bytes,
                                  csa2_stream_t stream) {
  g_last_launches = 0;
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  int launches = 0;
  const csa2_status s = run_pool(block_scores, n_vis, batch, n_max, params, pool_blocks, ws, ws_bytes,
                                 reinterpret_cast<cudaStream_t>(stream), &launches);
  if (s == CSA2_OK) g_last_launches = launches;
  return s;
}

csa2_status csa2_sparse_attn(const csa2_params *params, int32_t batch, const void *q, const uint8_t *kv, int64_t cap,
                             const int32_t *topk_idx, const uint8_t *swa, const float *swa_scale,
                             const int32_t *swa_len, float *out, float *lse, void *ws, size_t ws_bytes,
                             csa2_stream_t stream) {
  g_last_launches = 0;
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  int launches = 0;
  const csa2_status s = run_attn(params, batch, q, kv, cap, topk_idx, swa, swa_scale, swa_len, out, lse, ws, ws_bytes,
                                 reinterpret_cast<cudaStream_t>(stream), &launches);
  if (s == CSA2_OK) g_last_launches = launches;
  return s;
}

csa2_status csa2_sparse_decode(csa2_mode mode, const csa2_params *params, int32_t batch, const void *q,
                               const void *q_idx, const float *w, const uint8_t *kv, const void *k_idx, int64_t cap,
                               const int32_t *n_vis, int64_t n_max, const uint8_t *swa, const float *swa_scale,
                               const int32_t *swa_len, int32_t *topk_idx, int32_t *pool_blocks, float *out,
                               float *lse, void *ws, size_t ws_bytes, csa2_stream_t stream) {
  g_last_launches = 0;
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  if (mode != CSA2_MODE_FULL && mode != CSA2_MODE_REINDEX && mode != CSA2_MODE_REUSE) return CSA2_ERR_INVALID_ARG;
  if (batch < 1 || n_max < 0 || !ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) return CSA2_ERR_INVALID_ARG;
  if (ws_bytes < decode_ws(batch, n_max, params)) return CSA2_ERR_WORKSPACE;
  if ((mode == CSA2_MODE_REINDEX || (mode == CSA2_MODE_FULL && params->hsi)) && !pool_blocks)
    return CSA2_ERR_INVALID_ARG;
  if (mode != CSA2_MODE_REUSE && (!q_idx || !w || !k_idx || !n_vis)) return CSA2_ERR_INVALID_ARG;
  if (!q || !kv || !topk_idx || !out) return CSA2_ERR_INVALID_ARG;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  const int64_t nblk = (n_max + BLOCK - 1) / BLOCK;
  const size_t bs_bytes = (size_t)round_up((int64_t)batch * nblk * 4, 256);
  float *bscores = reinterpret_cast<float *>(wsb);
  uint8_t *rest = wsb + bs_bytes;   // the indexer's workspace, its histograms first
  const size_t rest_bytes = ws_bytes - bs_bytes;
  uint8_t *after_hist = rest + hist_ws(batch);   // the pool selection's and the readout's scratch
  const size_t after_bytes = rest_bytes - hist_ws(batch);
  int launches = 0;
  csa2_status s = CSA2_OK;
  if (mode == CSA2_MODE_FULL) {
    s = run_indexer(q_idx, w, k_idx, batch, cap, n_vis, n_max, nullptr, params, topk_idx,
                    params->hsi ? bscores : nullptr, rest, rest_bytes, st, &launches);
    if (s == CSA2_OK && params->hsi)
      s = run_pool(bscores, n_vis, batch, n_max, params, pool_blocks, after_hist, after_bytes, st, &launches);
  } else if (mode == CSA2_MODE_REINDEX) {
    s = run_indexer(q_idx, w, k_idx, batch, cap, n_vis, n_max, pool_blocks, params, topk_idx, nullptr, rest,
                    rest_bytes, st, &launches);
  }
  if (s == CSA2_OK)
    s = run_attn(params, batch, q, kv, cap, topk_idx, swa, swa_scale, swa_len, out, lse, after_hist, after_bytes, st,
                 &launches);
  if (s == CSA2_OK) g_last_launches = launches;
  return s;
}

}  // extern "C"

extern "C" csa2_status csa2_prefill_chunk(const csa2_params *params, int32_t batch, int32_t n_tokens, int64_t first_pos,
                                          int32_t m, const void *q, const void *q_idx, const float *w,
                                          const uint8_t *kv, const void *k_idx, int64_t cap, const uint8_t *swa,
                                          const float *swa_scale, int64_t swa_rows, int64_t swa_first_pos,
                                          int32_t *topk_idx, float *out, float *lse, void *ws, size_t ws_bytes,
                                          csa2_stream_t stream) {
  g_last_launches = 0;
  if (!params_ok(params)) return CSA2_ERR_UNSUPPORTED;
  if (params->indexer_fp4) return CSA2_ERR_UNSUPPORTED;   // the MXFP4 indexer is decode-only
  const csa2_params *p = params;
  if (batch < 1 || n_tokens < 8 || n_tokens % 8 != 0 || (m != 1 && m != 2) || first_pos < 0 || cap < 1)
    return CSA2_ERR_INVALID_ARG;
  if (!q || !q_idx || !w || !kv || !k_idx || !topk_idx || !out || !ws) return CSA2_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(q_idx) || !aligned16(w) || !aligned16(kv) || !aligned16(k_idx) ||
      (reinterpret_cast<uintptr_t>(ws) & 255u))
    return CSA2_ERR_INVALID_ARG;
  const int64_t last_pos = first_pos + n_tokens - 1;
  if ((last_pos + 1) / m > cap) return CSA2_ERR_INVALID_ARG;   // the chunk's entries must be in the cache
  const int W = p->sliding_window;
  if (W > 0) {
    if (!swa || !swa_scale || !aligned16(swa) || swa_first_pos < 0) return CSA2_ERR_INVALID_ARG;
    const int64_t first_start = first_pos - W + 1 > 0 ? first_pos - W + 1 : 0;
    if (first_start < swa_first_pos || last_pos - swa_first_pos >= swa_rows) return CSA2_ERR_INVALID_ARG;
  }
  const int64_t total = (int64_t)batch * n_tokens;
  if (total * HI >= ((int64_t)1 << 31) || (int64_t)batch * cap >= ((int64_t)1 << 31)) return CSA2_ERR_UNSUPPORTED;
  if (ws_bytes < prefill_ws(batch, cap, p)) return CSA2_ERR_WORKSPACE;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  const size_t scores_bytes = (size_t)round_up(kPrefillBlock * round_up(cap, SWEEP_TILE) * 4, 256);
  float *scores = reinterpret_cast<float *>(wsb);
  void *attn_ws = wsb + scores_bytes;
  CUtensorMap tm_k, tm_q;
  if (!make_tmap_bf16_rows128(&tm_k, k_idx, (int64_t)batch * cap, SWEEP_TILE)) return CSA2_ERR_CUDA;
  if (!make_tmap_bf16_rows128(&tm_q, q_idx, total * HI, 256)) return CSA2_ERR_CUDA;
  auto visible = [&](int64_t i) {
    const int64_t n = (first_pos + i + 1) / m;
    return n < cap ? n : cap;
  };
  const int sms = num_sms();
  int launches = 0;
  for (int64_t q0 = 0; q0 < total; q0 += kPrefillBlock) {
    const int64_t nq = total - q0 < kPrefillBlock ? total - q0 : kPrefillBlock;
    // the most entries any token of the block sees: the last token of a sequence
    // if the block holds one, else the block's last token
    const bool holds_end = (q0 / n_tokens) != ((q0 + nq - 1) / n_tokens) || (q0 + nq) % n_tokens == 0;
    const int64_t nv_max = holds_end ? visible(n_tokens - 1) : visible((q0 + nq - 1) % n_tokens);
    const int32_t tiles = (int32_t)((nv_max + SWEEP_TILE - 1) / SWEEP_TILE);
    PrefillIdxArgs ia;
    ia.w = w;
    ia.scores = scores;
    ia.cap = cap;
    ia.row_len = (int64_t)tiles * SWEEP_TILE;
    ia.first_pos = first_pos;
    ia.tokens = n_tokens;
    ia.q0 = q0;
    ia.groups = nq / 8;
    int64_t rt = (tiles * ia.groups + 4 * sms - 1) / (4 * sms);   // about 4 items per SM
    if (rt < 16) rt = 16;
    if (rt > tiles) rt = tiles > 0 ? tiles : 1;
    ia.range_tiles = (int32_t)rt;
    ia.ranges = (int32_t)((tiles + rt - 1) / rt);
    ia.tiles = tiles;
    ia.m = m;
    if (launch_prefill_indexer(tm_k, tm_q, ia, sms, st, &launches) != cudaSuccess) return CSA2_ERR_CUDA;
    TopkRows r;
    r.vals = scores;
    r.row_len = ia.row_len;
    r.row_stride = ia.row_len;
    r.rows = (int32_t)nq;
    r.k = p->index_topk;
    r.force_nvis = nullptr;
    r.force_block = BLOCK;
    r.n_max = cap;
    r.pool = nullptr;
    r.pool_stride = 0;
    r.out = topk_idx + q0 * p->index_topk;
    if (launch_topk(r, st, &launches) != cudaSuccess) return CSA2_ERR_CUDA;
    AttnArgs a;
    std::memset(&a, 0, sizeof(a));
    a.q = static_cast<const __nv_bfloat16 *>(q);
    a.kv = kv;
    a.idx = topk_idx;
    a.swa = swa;
    a.swa_scale = swa_scale;
    a.swa_len = nullptr;
    a.out = out;
    a.lse = lse;
    a.cap = cap;
    a.problems = (int32_t)nq;
    a.K = p->index_topk;
    a.W = W;
    a.kernel = p->attn_kernel;
    a.p0 = q0;
    a.tokens = n_tokens;
    a.causal_swa = 1;
    a.first_pos = first_pos;
    a.swa_first_pos = swa_first_pos;
    a.swa_seq_rows = swa_rows;
    if (launch_sparse_attn(a, attn_ws, st, &launches) != cudaSuccess) return CSA2_ERR_CUDA;
  }
  g_last_launches = launches;
  return CSA2_OK;
}
