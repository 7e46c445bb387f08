// CUDA-core (fp32 FMA) kernels: the float32 path of the norm estimators, the
// exact ghost-clipping norm, and the deterministic per-sample finish.
//
// The float32 path serves float32 inputs and shapes the tensor-core kernels
// do not take (odd widths, projection widths other than 16/32/64); it runs the
// same two contractions (sketch W = X R, then Y = X^T W) with fp32 operands.

#include <cuda_bf16.h>

#include "internal.h"

namespace dprc {
namespace {

template <typename T>
__device__ __forceinline__ float ld_f32(const T* p);
template <>
__device__ __forceinline__ float ld_f32<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_f32<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// W[i][t][j] = sum_c X[i][t][c] R[i?][c][j].  Block: 32 tokens x 64 columns,
// 256 threads, each thread 8 tokens of one column.  grid (ceil(T/32),
// ceil(n/64), B).
template <typename TX, typename TR>
__global__ void __launch_bounds__(256) simt_rowproj_kernel(const TX* __restrict__ X,
                                                           const TR* __restrict__ R,
                                                           long long r_bstride, int T, int c,
                                                           int n, float* __restrict__ W) {
  __shared__ float xs[32][33];
  __shared__ float rs[32][64];
  const int i = blockIdx.z, t0 = blockIdx.x * 32, j0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
  const TX* xi = X + static_cast<size_t>(i) * T * c;
  const TR* ri = R + static_cast<size_t>(i) * r_bstride;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int c0 = 0; c0 < c; c0 += 32) {
    for (int e = threadIdx.x; e < 32 * 32; e += 256) {
      const int tt = e >> 5, cc = e & 31;
      xs[tt][cc] = (t0 + tt < T && c0 + cc < c)
                       ? ld_f32(xi + static_cast<size_t>(t0 + tt) * c + c0 + cc)
                       : 0.f;
    }
    for (int e = threadIdx.x; e < 32 * 64; e += 256) {
      const int cc = e >> 6, jj = e & 63;
      rs[cc][jj] = (c0 + cc < c && j0 + jj < n)
                       ? ld_f32(ri + static_cast<size_t>(c0 + cc) * n + j0 + jj)
                       : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int cc = 0; cc < 32; ++cc) {
      const float r = rs[cc][tx];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(xs[ty * 8 + q][cc], r, acc[q]);
    }
    __syncthreads();
  }
  const int j = j0 + tx;
  if (j < n) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int t = t0 + ty * 8 + q;
      if (t < T) W[(static_cast<size_t>(i) * T + t) * n + j] = acc[q];
    }
  }
}

// Y[i][a][j] = sum_t X[i][t][a] W[i][t][j].  Block: 32 rows a x 64 columns.
// grid (ceil(c/32), ceil(n/64), B).
template <typename TX>
__global__ void __launch_bounds__(256) simt_colproj_kernel(const TX* __restrict__ X,
                                                           const float* __restrict__ W, int T,
                                                           int c, int n, float* __restrict__ Y) {
  __shared__ float xs[32][33];
  __shared__ float ws[32][64];
  const int i = blockIdx.z, a0 = blockIdx.x * 32, j0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 63, ty = threadIdx.x >> 6;
  const TX* xi = X + static_cast<size_t>(i) * T * c;
  const float* wi = W + static_cast<size_t>(i) * T * n;
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  for (int t0 = 0; t0 < T; t0 += 32) {
    for (int e = threadIdx.x; e < 32 * 32; e += 256) {
      const int tt = e >> 5, aa = e & 31;
      xs[tt][aa] = (t0 + tt < T && a0 + aa < c)
                       ? ld_f32(xi + static_cast<size_t>(t0 + tt) * c + a0 + aa)
                       : 0.f;
    }
    for (int e = threadIdx.x; e < 32 * 64; e += 256) {
      const int tt = e >> 6, jj = e & 63;
      ws[tt][jj] = (t0 + tt < T && j0 + jj < n) ? wi[static_cast<size_t>(t0 + tt) * n + j0 + jj]
                                                : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int tt = 0; tt < 32; ++tt) {
      const float w = ws[tt][tx];
#pragma unroll
      for (int q = 0; q < 8; ++q) acc[q] = fmaf(xs[tt][ty * 8 + q], w, acc[q]);
    }
    __syncthreads();
  }
  const int j = j0 + tx;
  if (j < n) {
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int a = a0 + ty * 8 + q;
      if (a < c) Y[(static_cast<size_t>(i) * c + a) * n + j] = acc[q];
    }
  }
}

// Deterministic block sum (fixed tree) of one float per thread; result in
// thread 0.  blockDim.x must be 256.
__device__ __forceinline__ float block_sum_256(float v, float* red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
  if (threadIdx.x == 0) {
    s = ((red[0] + red[1]) + (red[2] + red[3])) + ((red[4] + red[5]) + (red[6] + red[7]));
  }
  __syncthreads();
  return s;
}

// n[i] (+)= sum_{a,j} w_j Y[i][a][j]^2, one block per sample, fixed order.
__global__ void __launch_bounds__(256) simt_norm_finish_kernel(const float* __restrict__ Y,
                                                               long long c, int n, int n_head,
                                                               float w_tail,
                                                               float* __restrict__ n_out,
                                                               int accumulate) {
  __shared__ float red[8];
  const int i = blockIdx.x;
  const float* yi = Y + static_cast<size_t>(i) * c * n;
  const long long total = c * n;
  float s = 0.f;
  for (long long e = threadIdx.x; e < total; e += 256) {
    const float y = yi[e];
    const int j = static_cast<int>(e % n);
    s = fmaf((j < n_head ? 1.f : w_tail) * y, y, s);
  }
  s = block_sum_256(s, red);
  // a squared norm is never negative: a ghost-form sum that rounding in heavy
  // cancellation took below zero is returned as 0 (a NaN stays NaN)
  if (s < 0.f) s = 0.f;
  if (threadIdx.x == 0) n_out[i] = (accumulate ? n_out[i] : 0.f) + s;
}

// Exact norm by the ghost identity: per sample, the pair of 32-token tiles
// (tb, sb), tb <= sb, contributes w * sum_{t in tb, s in sb} (A A^T)_{ts}
// (G G^T)_{ts}, w = 1 on the diagonal and 2 off it (the two Grams are
// symmetric).  grid (ntiles, ntiles, B); blocks with sb < tb write 0.
template <typename TX>
__global__ void __launch_bounds__(256) exact_ghost_kernel(const TX* __restrict__ A,
                                                          const TX* __restrict__ G, int T,
                                                          int d, int p, int ntiles,
                                                          float* __restrict__ partials) {
  __shared__ float ta[32][33];
  __shared__ float sa[32][33];
  __shared__ float red[8];
  const int tb = blockIdx.x, sb = blockIdx.y, i = blockIdx.z;
  float* slot = partials + (static_cast<size_t>(i) * ntiles + tb) * ntiles + sb;
  if (sb < tb) {
    if (threadIdx.x == 0) *slot = 0.f;
    return;
  }
  // thread -> 4 entries (r, s0..s0+3) of the 32 x 32 Gram tile
  const int r = threadIdx.x >> 3, s0 = (threadIdx.x & 7) * 4;
  float ga[4] = {0.f, 0.f, 0.f, 0.f}, gg[4] = {0.f, 0.f, 0.f, 0.f};
  for (int pass = 0; pass < 2; ++pass) {
    const TX* X = pass == 0 ? A : G;
    const int w = pass == 0 ? d : p;
    const TX* xi = X + static_cast<size_t>(i) * T * w;
    float* acc = pass == 0 ? ga : gg;
    for (int k0 = 0; k0 < w; k0 += 32) {
      for (int e = threadIdx.x; e < 32 * 32; e += 256) {
        const int rr = e >> 5, kk = e & 31;
        const int t = tb * 32 + rr, s = sb * 32 + rr;
        const bool kin = k0 + kk < w;
        ta[rr][kk] = (t < T && kin) ? ld_f32(xi + static_cast<size_t>(t) * w + k0 + kk) : 0.f;
        sa[rr][kk] = (s < T && kin) ? ld_f32(xi + static_cast<size_t>(s) * w + k0 + kk) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        const float x = ta[r][kk];
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = fmaf(x, sa[s0 + q][kk], acc[q]);
      }
      __syncthreads();
    }
  }
  float v = 0.f;
#pragma unroll
  for (int q = 0; q < 4; ++q) v = fmaf(ga[q], gg[q], v);
  v = block_sum_256(v, red);
  if (threadIdx.x == 0) *slot = (tb == sb ? 1.f : 2.f) * v;
}

__global__ void __launch_bounds__(256) exact_finish_kernel(const float* __restrict__ partials,
                                                           long long per_sample,
                                                           float* __restrict__ n_out,
                                                           int accumulate) {
  __shared__ float red[8];
  const int i = blockIdx.x;
  const float* pi = partials + static_cast<size_t>(i) * per_sample;
  float s = 0.f;
  for (long long e = threadIdx.x; e < per_sample; e += 256) s += pi[e];
  s = block_sum_256(s, red);
  // a squared norm is never negative: a ghost-form sum that rounding in heavy
  // cancellation took below zero is returned as 0 (a NaN stays NaN)
  if (s < 0.f) s = 0.f;
  if (threadIdx.x == 0) n_out[i] = (accumulate ? n_out[i] : 0.f) + s;
}

template <typename TX, typename TR>
cudaError_t rowproj_t(const void* X, int64_t B, int64_t T, int64_t c, const void* R,
                      bool r_batched, int n, float* W, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>((T + 31) / 32), static_cast<unsigned>((n + 63) / 64),
            static_cast<unsigned>(B));
  simt_rowproj_kernel<TX, TR><<<grid, 256, 0, s>>>(
      static_cast<const TX*>(X), static_cast<const TR*>(R), r_batched ? c * n : 0,
      static_cast<int>(T), static_cast<int>(c), n, W);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_simt_rowproj(const void* X, dprc_dtype xdt, int64_t B, int64_t T, int64_t c,
                                const void* R, dprc_dtype rdt, bool r_batched, int n, float* W,
                                cudaStream_t s) {
  if (xdt == DPRC_F32 && rdt == DPRC_F32)
    return rowproj_t<float, float>(X, B, T, c, R, r_batched, n, W, s);
  if (xdt == DPRC_BF16 && rdt == DPRC_BF16)
    return rowproj_t<__nv_bfloat16, __nv_bfloat16>(X, B, T, c, R, r_batched, n, W, s);
  if (xdt == DPRC_BF16 && rdt == DPRC_F32)
    return rowproj_t<__nv_bfloat16, float>(X, B, T, c, R, r_batched, n, W, s);
  return rowproj_t<float, __nv_bfloat16>(X, B, T, c, R, r_batched, n, W, s);
}

cudaError_t launch_simt_colproj(const void* X, dprc_dtype xdt, int64_t B, int64_t T, int64_t c,
                                const float* W, int n, float* Y, cudaStream_t s) {
  dim3 grid(static_cast<unsigned>((c + 31) / 32), static_cast<unsigned>((n + 63) / 64),
            static_cast<unsigned>(B));
  if (xdt == DPRC_F32)
    simt_colproj_kernel<float><<<grid, 256, 0, s>>>(static_cast<const float*>(X), W,
                                                     static_cast<int>(T), static_cast<int>(c), n,
                                                     Y);
  else
    simt_colproj_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(X), W, static_cast<int>(T), static_cast<int>(c), n, Y);
  return cudaGetLastError();
}

cudaError_t launch_simt_norm_finish(const float* Y, int64_t B, int64_t c, int n, int n_head,
                                    float w_tail, float* n_out, int accumulate, cudaStream_t s) {
  simt_norm_finish_kernel<<<static_cast<unsigned>(B), 256, 0, s>>>(Y, c, n, n_head, w_tail, n_out,
                                                                    accumulate);
  return cudaGetLastError();
}

cudaError_t launch_partials_finish(const float* partials, int64_t B, int64_t per_sample,
                                   float* n_out, int accumulate, cudaStream_t s) {
  exact_finish_kernel<<<static_cast<unsigned>(B), 256, 0, s>>>(
      partials, static_cast<long long>(per_sample), n_out, accumulate);
  return cudaGetLastError();
}

cudaError_t launch_exact_ghost(const void* A, const void* G, dprc_dtype dt, int64_t B,
                               int64_t T, int64_t d, int64_t p, float* partials, float* n_out,
                               int accumulate, cudaStream_t s) {
  const int ntiles = static_cast<int>((T + 31) / 32);
  dim3 grid(ntiles, ntiles, static_cast<unsigned>(B));
  if (dt == DPRC_F32)
    exact_ghost_kernel<float><<<grid, 256, 0, s>>>(
        static_cast<const float*>(A), static_cast<const float*>(G), static_cast<int>(T),
        static_cast<int>(d), static_cast<int>(p), ntiles, partials);
  else
    exact_ghost_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(
        static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(G),
        static_cast<int>(T), static_cast<int>(d), static_cast<int>(p), ntiles, partials);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  exact_finish_kernel<<<static_cast<unsigned>(B), 256, 0, s>>>(
      partials, static_cast<long long>(ntiles) * ntiles, n_out, accumulate);
  return cudaGetLastError();
}

}  // namespace dprc
