// csa2_hier_pool_select_static: the HSI pool selection with its scratch in a
// fixed device array owned by this library instead of a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// pool selection: a runtime that replays a pre-planned memory layout and
// forbids allocation while it executes, or host code that only holds raw
// device pointers to its inputs and outputs and has no allocator of its own.
// For them this call takes no workspace argument and never calls cudaMalloc,
// cudaFree or any allocating routine.
//
// The scratch is kScratchBytes of static device memory; every GPU that loads
// this library holds it until the process exits.  Its device address is
// looked up once per device (cudaGetSymbolAddress, with that device current)
// on the first call made on that device, so that first call should happen
// before any stream capture.  All calls on a device share the one array and
// it keeps the last call's contents: the selection clears the counters it
// needs at the start of every call, and calls whose work overlaps on the GPU
// (different streams, or different host threads) race on it.
#include <mutex>

#include "kernels.cuh"

namespace csa2 {
namespace {

constexpr size_t kScratchBytes = CSA2_POOL_STATIC_SCRATCH_BYTES;   // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) uint8_t g_pool_scratch[kScratchBytes];

std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of the static scratch on the current device (set up once
// per device).
cudaError_t scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pool_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace
}  // namespace csa2

using namespace csa2;

extern "C" csa2_status csa2_hier_pool_select_static(const float *block_scores, const int32_t *n_vis,
                                                    int32_t batch, int64_t n_max, const csa2_params *params,
                                                    int32_t *pool_blocks, csa2_stream_t stream) {
  set_last_launch_count(0);
  if (!params || params->candidate_block_size != BLOCK || params->candidate_topk_blocks < 16 ||
      params->candidate_topk_blocks > TOPK_MAX_K || params->candidate_topk_blocks % 16 != 0)
    return CSA2_ERR_UNSUPPORTED;
  if (!block_scores || !n_vis || !pool_blocks || batch < 1 || n_max < 0) return CSA2_ERR_INVALID_ARG;
  const int64_t nblk = (n_max + BLOCK - 1) / BLOCK;
  const size_t need = topk_scratch_bytes(batch, nblk, params->candidate_topk_blocks);
  if (need > kScratchBytes) return CSA2_ERR_WORKSPACE;   // beyond the static scratch
  void *scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return CSA2_ERR_CUDA;
  TopkRows r;
  r.vals = block_scores;
  r.row_len = nblk;
  r.row_stride = nblk;
  r.rows = batch;
  r.k = params->candidate_topk_blocks;
  r.force_nvis = n_vis;
  r.force_block = BLOCK;
  r.n_max = n_max;
  r.pool = nullptr;
  r.pool_stride = 0;
  r.out = pool_blocks;
  int launches = 0;
  const cudaError_t e = launch_pool_topk(r, scratch, 0, reinterpret_cast<cudaStream_t>(stream), &launches);
  if (e != cudaSuccess) return CSA2_ERR_CUDA;
  set_last_launch_count(launches);
  return CSA2_OK;
}
