// csa2_kv_quant_write kernel: compressor (m = 2) -> RoPE on the tail 64
// channels -> FP4 (E2M1 codes, one E4M3 scale per 16 channels, no global
// scale).  "DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression",
// section 2.4.4 (quantisation after RoPE; E2M1 with an E4M3 scale per 16
// channels, no second-level scale); "DeepSeek-V4.1-Flash - Architecture",
// section 4.
//
// One warp writes one 288-byte entry; lane g owns channel group g (16
// channels): it loads 32 bytes of bf16 per source position, produces its
// scale byte and 8 bytes of codes, so the warp stores 256 contiguous code
// bytes and 32 contiguous scale bytes.  Decode writes one entry per sequence,
// so the kernel is latency-bound; the m = 2 chunked-prefill write streams
// 4 KB of input per entry and is bandwidth-bound.
//
// With a projection (csa2_kv_quant_write_ik) the same warp also writes the
// entry's indexer key: k = W_ik e over the entry before FP4 quantisation
// ("DeepSeek-v4.1 Flash: Pushing the Limits of KV Cache Compression", 2.3.1:
// the Indexer K is a projection of the main KV entry).  Each lane forms the
// partial dot products of its 16 channels with 32 rows of W_ik at a time
// (W_ik read as 32-byte row pieces, one per lane, coalesced), a transposed
// warp reduction leaves row 32g + l on lane l (four warps per entry, one per
// block of 32 rows; warps 1-3 stage W_ik in shared memory while warp 0
// computes the entry), and the row is stored as bf16
// (round to nearest even) or, for the MXFP4 indexer, quantised per block of
// 32 (one block per group of 32 rows) exactly like csa2_indexer_k_quant.
#include <cmath>

#include "kernels.cuh"

namespace csa2 {

namespace {

struct RopeFreqs {
  float inv[ROPE_DIM / 2];
};

// Positions must stay below 2^22 so that the 2*pi reduction stays exact.
constexpr int64_t kMaxRopePos = int64_t(1) << 22;

__device__ __forceinline__ void load_bf16x16(const __nv_bfloat16 *p, float (&x)[16]) {
  const uint4 *v = reinterpret_cast<const uint4 *>(p);
  uint4 a = __ldg(v), b = __ldg(v + 1);
  uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Cody-Waite split of 2*pi: C1 and C2 carry 33 significant bits each, so
// k * C1 and k * C2 are exact for k < 2^20; C1 + C2 + C3 = 2*pi to about
// 2^-120 (the three parts were derived with 300-bit arithmetic).
constexpr double kTwoPi1 = 0x1.921fb544p+2;
constexpr double kTwoPi2 = 0x1.0b4611a6p-32;
constexpr double kTwoPi3 = 0x1.3198a2e037073p-67;
constexpr double kInvTwoPi = 0.15915494309189535;

// The indexer-key output of the projecting write.
struct IkOut {
  const __nv_bfloat16 *w;   // W_ik [128][512]
  void *k;                  // bf16 [k_rows][128], or the MXFP4 planes of k_rows rows
  int64_t k_rows;
  int fp4;
};

// One halving step of the transposed reduction: lanes with bit HALF set keep
// the upper N of their 2N columns and add the partner's, the others the
// lower N.
template <int N, int HALF>
__device__ __forceinline__ void reduce_step(float (&x)[32], int lane) {
  const bool up = lane & HALF;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    const float send = up ? x[i] : x[i + N];
    const float keep = up ? x[i + N] : x[i];
    x[i] = keep + __shfl_xor_sync(0xffffffffu, send, HALF);
  }
}

// Sum over the 32 lanes of each of 32 columns: lane l returns column l.
__device__ __forceinline__ float transpose_reduce32(float (&x)[32], int lane) {
  reduce_step<16, 16>(x, lane);
  reduce_step<8, 8>(x, lane);
  reduce_step<4, 4>(x, lane);
  reduce_step<2, 2>(x, lane);
  reduce_step<1, 1>(x, lane);
  return x[0];
}

// 16 bf16 from shared memory as floats.
__device__ __forceinline__ void lds_bf16x16(const __nv_bfloat16 *p, float (&x)[16]) {
  const uint4 *v = reinterpret_cast<const uint4 *>(p);
  uint4 a = v[0], b = v[1];
  uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

// Rows 32g .. 32g + 31 of k = W_ik e for the entry whose channels 16 lane ..
// +15 this lane holds in x (W_ik staged in shared memory as w_s), stored at
// row `row` of the indexer-K cache.
__device__ __forceinline__ void project_indexer_block(const IkOut &ik, const __nv_bfloat16 *w_s, const float (&x)[16],
                                                      int lane, int64_t row, int g) {
  const int c0 = lane * 16;
  float part[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    float wv[16];
    lds_bf16x16(w_s + (g * 32 + j) * D + c0, wv);
    float acc = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) acc = fmaf(wv[i], x[i], acc);
    part[j] = acc;
  }
  const __nv_bfloat16 kb = __float2bfloat16_rn(transpose_reduce32(part, lane));   // row 32 g + lane
  if (!ik.fp4) {
    static_cast<__nv_bfloat16 *>(ik.k)[row * DI + g * 32 + lane] = kb;
    return;
  }
  // MXFP4 block g: E = floor(log2 max|k|) - 2 in [-127, 127] (-127 for a
  // zero or subnormal maximum), codes E2M1_rne_satfinite(k / 2^E)
  const float v = __bfloat162float(kb);
  float am = fabsf(v);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
  const int ef = (int)((__float_as_uint(am) >> 23) & 0xFFu);
  const int E = (am > 0.0f && ef > 0) ? max(-127, min(127, ef - 127 - 2)) : -127;
  const float inv = -E >= -126 ? __uint_as_float((uint32_t)(-E + 127) << 23) : __uint_as_float(0x00400000u);
  const float partner = __shfl_xor_sync(0xffffffffu, v, 1);
  uint8_t *planes = static_cast<uint8_t *>(ik.k);
  if ((lane & 1) == 0)   // element 2j (this lane) in the low nibble, 2j + 1 in the high one
    planes[row * (DI / 2) + g * 16 + (lane >> 1)] = (uint8_t)cvt_e2m1x2(partner * inv, v * inv);
  if (lane == 0) planes[ik.k_rows * (DI / 2) + row * 4 + g] = (uint8_t)(E + 127);
}

template <bool kProject>
__global__ void __launch_bounds__(256) kv_quant_write_kernel(const __nv_bfloat16 *__restrict__ latent,
                                                             const __nv_bfloat16 *__restrict__ z, int m,
                                                             int64_t n_entries, const int64_t *__restrict__ pos,
                                                             const int64_t *__restrict__ slot,
                                                             uint8_t *__restrict__ kv, int64_t kv_rows,
                                                             const RopeFreqs freqs, const IkOut ik) {
  pdl_wait();   // the inputs' producer is complete past here (programmatic launch)
  const int lane = threadIdx.x & 31;
  // one entry per warp; when projecting, one entry per block of 4 warps:
  // warp 0 writes the entry, then each warp projects 32 rows of W_ik
  const int64_t e = kProject ? (int64_t)blockIdx.x : (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (e >= n_entries) return;   // uniform over the warp (the block, when projecting)
  const int64_t row = slot[e];
  const int64_t p = pos[e];
  if (row < 0 || row >= kv_rows || p < 0 || p >= kMaxRopePos || (kProject && row >= ik.k_rows)) {
    if (lane == 0 && (!kProject || threadIdx.x == 0)) set_error(CSA2_DEV_ERR_INDEX);
    return;
  }
  __shared__ float e_s[kProject ? D : 1];
  extern __shared__ __align__(16) uint8_t w_dyn[];   // projecting: W_ik [128][512] bf16
  const __nv_bfloat16 *w_s = reinterpret_cast<const __nv_bfloat16 *>(w_dyn);
  if (kProject && threadIdx.x >= 32) {
    // warps 1..3 stage W_ik while warp 0 computes the entry
    // (asynchronous 16-byte copies: all of a thread's copies in flight)
    const uint4 *src = reinterpret_cast<const uint4 *>(ik.w);
    uint4 *dst = reinterpret_cast<uint4 *>(w_dyn);
    for (int i = threadIdx.x - 32; i < DI * D / 8; i += blockDim.x - 32) cp_async16(dst + i, src + i);
    cp_async_commit();
    cp_async_wait_all();
    __syncthreads();   // the entry is in e_s, W_ik in w_dyn
    float x[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) x[i] = e_s[lane * 16 + i];
    project_indexer_block(ik, w_s, x, lane, row, threadIdx.x >> 5);
    return;
  }
  // Lane j evaluates the rotation of pair j: angle = pos * inv_freq_j (exact
  // in double), reduced modulo 2*pi (Cody-Waite, k < 2^20), cos / sin in
  // double, rounded to fp32.
  float cj, sj;
  {
    const double ang = (double)p * (double)freqs.inv[lane];
    const double k = rint(ang * kInvTwoPi);
    double r = fma(-k, kTwoPi1, ang);
    r = fma(-k, kTwoPi2, r);
    r = fma(-k, kTwoPi3, r);
    double sd, cd;
    sincos(r, &sd, &cd);
    cj = __double2float_rn(cd);
    sj = __double2float_rn(sd);
  }
  const int c0 = lane * 16;
  float x[16];
  if (m == 1) {
    load_bf16x16(latent + e * D + c0, x);
  } else {
    // Channel-wise softmax over the m = 2 source positions, in double,
    // rounded once to fp32.
    float x0[16], x1[16], z0[16], z1[16];
    load_bf16x16(latent + (e * 2 + 0) * D + c0, x0);
    load_bf16x16(latent + (e * 2 + 1) * D + c0, x1);
    load_bf16x16(z + (e * 2 + 0) * D + c0, z0);
    load_bf16x16(z + (e * 2 + 1) * D + c0, z1);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      // explicit IEEE double ops: no contraction into fused multiply-adds.
      // The larger logit's exponent is exp(0) = 1 exactly, so only the other
      // one is evaluated, and its weight 1 / den is the correctly rounded
      // reciprocal (the same values as two exps and two divisions).
      const double zm = fmax((double)z0[i], (double)z1[i]);
      const bool first = (double)z0[i] >= (double)z1[i];
      const double eo = exp(__dsub_rn(first ? (double)z1[i] : (double)z0[i], zm));
      const double den = __dadd_rn(1.0, eo);
      const double w_one = __drcp_rn(den), w_other = __ddiv_rn(eo, den);
      const double wa = first ? w_one : w_other, wb = first ? w_other : w_one;
      const double num = __dadd_rn(__dmul_rn(wa, (double)x0[i]), __dmul_rn(wb, (double)x1[i]));
      x[i] = __double2float_rn(num);
    }
  }
  // RoPE: interleaved pairs (448 + 2j, 449 + 2j); lanes 28..31 own channels
  // 448..511 and take the 8 rotations they need from the lanes that computed
  // them; products and sums rounded separately (no fused multiply-add).
  const int jbase = (lane - (D - ROPE_DIM) / 16) * 8;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int src = (jbase + i) & 31;
    const float c = __shfl_sync(0xffffffffu, cj, src);
    const float s = __shfl_sync(0xffffffffu, sj, src);
    if (c0 >= D - ROPE_DIM) {
      const float a = x[2 * i], b = x[2 * i + 1];
      x[2 * i] = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, s));
      x[2 * i + 1] = __fadd_rn(__fmul_rn(a, s), __fmul_rn(b, c));
    }
  }
  if (kProject) {
#pragma unroll
    for (int i = 0; i < 16; ++i) e_s[lane * 16 + i] = x[i];
    __syncthreads();
    project_indexer_block(ik, w_s, x, lane, row, 0);
  }
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint32_t sbyte = cvt_e4m3(__fdiv_rn(amax, 6.0f));
  const float sd = e4m3_to_f32(sbyte);
  uint32_t lo = 0, hi = 0;
  if (sd != 0.0f) {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      lo |= cvt_e2m1x2(__fdiv_rn(x[2 * i + 1], sd), __fdiv_rn(x[2 * i], sd)) << (8 * i);
      hi |= cvt_e2m1x2(__fdiv_rn(x[8 + 2 * i + 1], sd), __fdiv_rn(x[8 + 2 * i], sd)) << (8 * i);
    }
  }
  uint8_t *dst = kv + row * ENTRY_BYTES;
  reinterpret_cast<uint2 *>(dst)[lane] = make_uint2(lo, hi);
  dst[256 + lane] = (uint8_t)sbyte;
}

}  // namespace

cudaError_t launch_kv_quant_write(const void *latent, const void *z, int m, int64_t n_entries, const int64_t *pos,
                                  const int64_t *slot, uint8_t *kv, int64_t kv_rows, float rope_theta,
                                  cudaStream_t stream, const void *w_ik, void *k_out, int64_t k_rows, int fp4) {
  // inverse frequencies fl32(theta^(-2j/64)), j = 0..31, evaluated on the host
  RopeFreqs freqs;
  for (int j = 0; j < ROPE_DIM / 2; ++j)
    freqs.inv[j] = (float)std::pow((double)rope_theta, -(2.0 * j) / (double)ROPE_DIM);
  IkOut ik;
  ik.w = static_cast<const __nv_bfloat16 *>(w_ik);
  ik.k = k_out;
  ik.k_rows = k_rows;
  ik.fp4 = fp4;
  // Few entries (decode): one warp per block, so that the double-precision
  // rotations of different entries run on different SMs (FP64 throughput per
  // SM is low); many entries: 8 warps per block.
  const int warps = n_entries <= 1024 ? 1 : 8;
  const int64_t blocks = (n_entries + warps - 1) / warps;
  if (w_ik) {
    const int smem = DI * D * 2;   // W_ik staged per block
    cudaError_t err = cudaFuncSetAttribute(kv_quant_write_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           smem);
    if (err != cudaSuccess) return err;
    return launch_pdl(kv_quant_write_kernel<true>, dim3((unsigned)n_entries), dim3((DI / 32) * 32), smem, stream, 0u,
                      static_cast<const __nv_bfloat16 *>(latent), static_cast<const __nv_bfloat16 *>(z), m, n_entries,
                      pos, slot, kv, kv_rows, freqs, ik);
  }
  return launch_pdl(kv_quant_write_kernel<false>, dim3((unsigned)blocks), dim3(warps * 32), 0, stream, 0u,
                    static_cast<const __nv_bfloat16 *>(latent), static_cast<const __nv_bfloat16 *>(z), m, n_entries,
                    pos, slot, kv, kv_rows, freqs, ik);
}

}  // namespace csa2
