// Clip factors and the Gaussian noise add of DP-SGD-RC.
//
// Clip (papernotes.org, "Method > Overall framework"): each sample's loss is
// rescaled by c_i = min(1, C / sqrt(n_i)), n_i the layerwise sum of the
// squared-norm estimates.
//
// Noise (same section; the aggregated gradient receives sigma*C*N(0, I)):
// normals come from the counter-based Philox4x32-10 generator of Salmon,
// Moraes, Dror and Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3"
// (SC'11), implemented here from that paper's definition, followed by the
// Box-Muller transform.  Stream layout: element e uses word (e & 3) of block
// e >> 2; block j = Philox(counter (j_lo, j_hi, step_lo, step_hi), key
// (seed_lo, seed_hi)).  The kernel is HBM-bound: 8 bytes of traffic per
// element (read + write of the fp32 gradient), read with 128-bit loads.

#include "common.cuh"
#include "internal.h"

namespace dprc {
namespace {

// -2 ln(u1) for u1 = m 2^-24, m = (a >> 8) + 1 in [1, 2^24].  The hardware
// logarithm (__logf, absolute error <= 2^-21.41 on [0.5, 2]) loses relative
// accuracy as u1 -> 1, so for v = 1 - u1 <= 2^-5 (v exact) the Taylor series
//   -ln(1 - v) = v (1 + v/2 + v^2/3 + ... + v^6/7)
// is used instead (truncation below 4e-12 relative).  Both are evaluated and
// one selected, so warps do not diverge.
__device__ __forceinline__ float neg2log_u1(uint32_t a) {
  const uint32_t m = (a >> 8) + 1u;
  const uint32_t w = (1u << 24) - m;  // 2^24 v
  const float v = static_cast<float>(w) * 5.9604644775390625e-8f;
  float t = 0.14285714285714285f;     // 1/7
  t = fmaf(t, v, 0.16666666666666666f);
  t = fmaf(t, v, 0.2f);
  t = fmaf(t, v, 0.25f);
  t = fmaf(t, v, 0.33333333333333333f);
  t = fmaf(t, v, 0.5f);
  t = fmaf(t, v, 1.0f);
  const float series = 2.0f * v * t;
  const float u1 = static_cast<float>(m) * 5.9604644775390625e-8f;
  const float hw = -2.0f * __logf(u1);
  return w <= (1u << 19) ? series : hw;
}

// Box-Muller on a word pair: u1 = ((a >> 8) + 1) 2^-24 in (0, 1],
// u2 = (b >> 8) 2^-24 in [0, 1):  (r cos 2 pi u2, r sin 2 pi u2),
// r = sqrt(-2 ln u1).  The angle is taken as x + pi with x = 2 pi (u2 - 1/2)
// in [-pi, pi), where the hardware sine and cosine have absolute error
// <= 2^-21.41, hence |error| <= 2e-6 + 1e-6 r for each normal.  r is taken as
// q rsqrt(q), q = -2 ln u1 (rsqrtf within 2 ulp: relative 2.5e-7 in r, inside
// that bound; a few instructions fewer than the correctly rounded sqrtf in a
// kernel whose instruction issue sits close to its memory time); q = 0
// (u1 = 1) gives r = 0.
__device__ __forceinline__ float2 box_muller(uint32_t a, uint32_t b) {
  const float q = neg2log_u1(a);
  const float rad = q > 0.f ? q * rsqrtf(q) : 0.f;
  const float t = static_cast<float>(b >> 8) * 5.9604644775390625e-8f - 0.5f;  // exact
  float s, c;
  __sincosf(6.283185307179586f * t, &s, &c);
  return make_float2(-rad * c, -rad * s);
}

__device__ __forceinline__ float4 add_noise4(float4 g, uint4 w, float scale) {
  const float2 z01 = box_muller(w.x, w.y);
  const float2 z23 = box_muller(w.z, w.w);
  g.x = fmaf(scale, z01.x, g.x);
  g.y = fmaf(scale, z01.y, g.y);
  g.z = fmaf(scale, z23.x, g.z);
  g.w = fmaf(scale, z23.y, g.w);
  return g;
}

// Each thread issues kNoiseUnroll 16-byte loads before any arithmetic, and
// the grid holds kNoiseCtasPerSm CTAs per SM (eight resident at a time) that
// stride over the buffer.  A sweep on GB300 (unroll 1-16, 128-512 threads,
// 8 CTAs per SM up to one CTA per tile) put the optimum at two loads per
// thread and 64-96 CTAs per SM: enough independent warps to hide the load
// latency behind the generator, without the register cost of deeper unrolls
// or the tail of one-tile CTAs.
constexpr int kNoiseUnroll = 2;
constexpr int kNoiseCtasPerSm = 64;

// grad[i] += scale z_{4 blk0 + i}: the fp32 buffer starts at a block boundary
// of the stream (blk0 = 0 for a whole gradient).
__global__ void __launch_bounds__(256) noise_kernel(float* __restrict__ grad, long long n,
                                                    float scale, uint64_t seed, uint64_t step,
                                                    uint64_t blk0) {
  const RoundKeys rk = round_keys(seed);
  const long long nblk = n >> 2;
  float4* g4 = reinterpret_cast<float4*>(grad);
  const long long tile = static_cast<long long>(blockDim.x) * kNoiseUnroll;
  for (long long base = static_cast<long long>(blockIdx.x) * tile; base < nblk;
       base += static_cast<long long>(gridDim.x) * tile) {
    float4 g[kNoiseUnroll];
#pragma unroll
    for (int u = 0; u < kNoiseUnroll; ++u) {
      const long long j = base + u * blockDim.x + threadIdx.x;
      if (j < nblk) g[u] = __ldcs(g4 + j);
    }
#pragma unroll
    for (int u = 0; u < kNoiseUnroll; ++u) {
      const long long j = base + u * blockDim.x + threadIdx.x;
      if (j < nblk)
        __stcs(g4 + j,
               add_noise4(g[u], philox_block(blk0 + static_cast<uint64_t>(j), step, rk), scale));
    }
  }
  // ragged tail: the last n & 3 elements, one thread
  if (blockIdx.x == 0 && threadIdx.x == 0 && (n & 3) != 0) {
    const uint4 w = philox_block(blk0 + static_cast<uint64_t>(nblk), step, rk);
    const float2 z01 = box_muller(w.x, w.y);
    const float2 z23 = box_muller(w.z, w.w);
    const float z[4] = {z01.x, z01.y, z23.x, z23.y};
    for (long long e = nblk * 4; e < n; ++e) grad[e] = fmaf(scale, z[e - nblk * 4], grad[e]);
  }
}

// The four normals of stream block q (words 0..3 as elements 4q .. 4q + 3).
__device__ __forceinline__ void block_normals(uint64_t q, uint64_t step, const RoundKeys& rk,
                                              float* z) {
  const uint4 w = philox_block(q, step, rk);
  const float2 z01 = box_muller(w.x, w.y);
  const float2 z23 = box_muller(w.z, w.w);
  z[0] = z01.x;
  z[1] = z01.y;
  z[2] = z23.x;
  z[3] = z23.y;
}

__device__ __forceinline__ float load_f(const float* p) { return *p; }
__device__ __forceinline__ float load_f(const __nv_bfloat16* p) { return __bfloat162float(*p); }
__device__ __forceinline__ void store_f(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_f(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// grad[i] += scale z_{e0 + i} for any element type TG (fp32 or bf16) and any
// stream offset e0 with e0 & 3 == R: a thread owns V consecutive elements (16
// bytes), whose stream positions span NB Philox blocks; the sum is formed in
// fp32 and rounded once to TG.  The last n mod V elements: one thread.
template <typename TG, int R>
__global__ void __launch_bounds__(256) noise_at_kernel(TG* __restrict__ grad, long long n,
                                                       float scale, uint64_t seed, uint64_t step,
                                                       uint64_t e0) {
  constexpr int V = 16 / static_cast<int>(sizeof(TG));
  constexpr int NB = (R + V + 3) / 4;
  const RoundKeys rk = round_keys(seed);
  const long long nvec = n / V;
  const uint64_t q0 = e0 >> 2;  // block of element 0
  uint4* g16 = reinterpret_cast<uint4*>(grad);
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long j = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; j < nvec;
       j += stride) {
    uint4 raw = __ldcs(g16 + j);
    TG* v = reinterpret_cast<TG*>(&raw);
    float z[4 * NB];
#pragma unroll
    for (int b = 0; b < NB; ++b)
      block_normals(q0 + static_cast<uint64_t>(j) * (V / 4) + b, step, rk, z + 4 * b);
#pragma unroll
    for (int t = 0; t < V; ++t) store_f(v + t, fmaf(scale, z[R + t], load_f(v + t)));
    __stcs(g16 + j, raw);
  }
  if (blockIdx.x == 0 && threadIdx.x == 0) {
    for (long long i = nvec * V; i < n; ++i) {
      float z[4];
      const uint64_t e = e0 + static_cast<uint64_t>(i);
      block_normals(e >> 2, step, rk, z);
      const int w = static_cast<int>(e & 3);
      const float ze = w == 0 ? z[0] : (w == 1 ? z[1] : (w == 2 ? z[2] : z[3]));
      store_f(grad + i, fmaf(scale, ze, load_f(grad + i)));
    }
  }
}

__global__ void __launch_bounds__(256) philox_words_kernel(uint4* __restrict__ out, long long n,
                                                           uint64_t first, uint64_t seed,
                                                           uint64_t step) {
  const RoundKeys rk = round_keys(seed);
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long j = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; j < n;
       j += stride)
    out[j] = philox_block(first + static_cast<uint64_t>(j), step, rk);
}

// Launched as a programmatic dependent of the norm kernel before it: the
// launch overlaps that kernel, and griddepcontrol.wait holds the reads of n
// until it has completed and its writes are visible.
// S [n] in {-1, +1} (n = p k, row-major [p][k]) as TO: entry e is bit (e & 31)
// of word (e >> 5) & 3 of Philox block e >> 7 of the stream of (seed, step);
// bit 1 gives -1.  One thread per block of 128 entries.
template <typename TO>
__global__ void __launch_bounds__(256) pm1_signs_kernel(TO* __restrict__ out, long long n,
                                                        uint64_t seed, uint64_t step) {
  const RoundKeys rk = round_keys(seed);
  const long long nblk = (n + 127) / 128;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long j = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; j < nblk;
       j += stride) {
    const uint4 w = philox_block(static_cast<uint64_t>(j), step, rk);
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
    for (int q = 0; q < 4; ++q)
      for (int b = 0; b < 32; ++b) {
        const long long e = j * 128 + q * 32 + b;
        if (e < n) out[e] = static_cast<TO>(((words[q] >> b) & 1u) ? -1.0f : 1.0f);
      }
  }
}

__global__ void clip_kernel(const float* __restrict__ n, long long B, float C,
                            float* __restrict__ c, int32_t* __restrict__ nonfinite) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= B) return;
  bool bad;
  c[i] = clip_factor(n[i], C, bad);
  if (bad && nonfinite != nullptr) atomicAdd(nonfinite, 1);
}

int grid_for(long long work, int threads, int ctas_per_sm = 8) {
  const int sms = device_sm_count();
  long long blocks = (work + threads - 1) / threads;
  const long long cap = static_cast<long long>(sms) * ctas_per_sm;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  return static_cast<int>(blocks);
}

}  // namespace

cudaError_t launch_noise(float* grad, int64_t N, float sigma, float C, uint64_t seed,
                         uint64_t step, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  noise_kernel<<<grid_for(N / 4 / kNoiseUnroll + 1, 256, kNoiseCtasPerSm), 256, 0, s>>>(
      grad, N, sigma * C, seed, step, 0);
  return cudaGetLastError();
}

namespace {
template <typename TG>
cudaError_t launch_noise_at_t(TG* grad, int64_t N, uint64_t e0, float scale, uint64_t seed,
                              uint64_t step, cudaStream_t s) {
  constexpr int V = 16 / static_cast<int>(sizeof(TG));
  const int grid = grid_for(N / V + 1, 256, kNoiseCtasPerSm);
  switch (e0 & 3) {
    case 0: noise_at_kernel<TG, 0><<<grid, 256, 0, s>>>(grad, N, scale, seed, step, e0); break;
    case 1: noise_at_kernel<TG, 1><<<grid, 256, 0, s>>>(grad, N, scale, seed, step, e0); break;
    case 2: noise_at_kernel<TG, 2><<<grid, 256, 0, s>>>(grad, N, scale, seed, step, e0); break;
    default: noise_at_kernel<TG, 3><<<grid, 256, 0, s>>>(grad, N, scale, seed, step, e0);
  }
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_noise_at(void* grad, dprc_dtype dt, int64_t N, uint64_t first_element,
                            float sigma, float C, uint64_t seed, uint64_t step, cudaStream_t s) {
  if (N == 0) return cudaSuccess;
  if (dt == DPRC_F32 && (first_element & 3) == 0) {
    // a block boundary: the whole-gradient kernel with its block offset
    noise_kernel<<<grid_for(N / 4 / kNoiseUnroll + 1, 256, kNoiseCtasPerSm), 256, 0, s>>>(
        static_cast<float*>(grad), N, sigma * C, seed, step, first_element >> 2);
    return cudaGetLastError();
  }
  if (dt == DPRC_F32)
    return launch_noise_at_t(static_cast<float*>(grad), N, first_element, sigma * C, seed, step,
                             s);
  return launch_noise_at_t(static_cast<__nv_bfloat16*>(grad), N, first_element, sigma * C, seed,
                           step, s);
}

cudaError_t launch_philox_words(uint32_t* out, int64_t n_blocks, uint64_t first_block,
                                uint64_t seed, uint64_t step, cudaStream_t s) {
  if (n_blocks == 0) return cudaSuccess;
  philox_words_kernel<<<grid_for(n_blocks, 256), 256, 0, s>>>(reinterpret_cast<uint4*>(out),
                                                              n_blocks, first_block, seed, step);
  return cudaGetLastError();
}

cudaError_t launch_pm1_signs(void* out, dprc_dtype dt, int64_t n, uint64_t seed, uint64_t step,
                             cudaStream_t s) {
  const int grid = grid_for((n + 127) / 128, 256);
  if (dt == DPRC_F32)
    pm1_signs_kernel<float><<<grid, 256, 0, s>>>(static_cast<float*>(out), n, seed, step);
  else
    pm1_signs_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(static_cast<__nv_bfloat16*>(out), n,
                                                         seed, step);
  return cudaGetLastError();
}

cudaError_t launch_clip(const float* n, int64_t B, float C, float* c, int32_t* nonfinite,
                        cudaStream_t s) {
  const int threads = 128;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((B + threads - 1) / threads));
  cfg.blockDim = dim3(threads);
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, clip_kernel, n, static_cast<long long>(B), C, c, nonfinite);
}

}  // namespace dprc
