// Hutch++ middle step (papernotes.org, "Key design > Hutch++ head-tail
// decomposition": Q is an orthonormal basis of Col(O S); the tail runs
// Hutchinson on the residual (I - Q Q^T)):
//
//   Q_i  = thin Q of a Householder QR of M_i = O_i S      (p x r, per sample)
//   P'_i = P - Q_i (Q_i^T P)
//
// and the concatenation [Q_i | P'_i] is written in the layout the next row
// projection reads.  One CTA per sample, fp32.  The estimate depends only on
// span(Q), so the columns of M are first rescaled by their largest magnitude
// (span unchanged), which keeps every sum of squares far from fp32 over- and
// underflow.  Householder QR stays orthonormal when M is rank deficient (a
// zero reflector is the identity), which is exactly the low-rank case where
// Hutch++ is exact.

#include <cuda_bf16.h>

#include "internal.h"

namespace dprc {
namespace {

constexpr int kQrThreads = 512;
constexpr int kQrWarps = kQrThreads / 32;
constexpr int kMaxR = 64;

// Reduces NV per-thread partial values across the block (fixed order).
// Result in out[0..NV).  op: 0 = sum, 1 = max.
template <int NV>
__device__ void block_reduce(float (&v)[NV], int nv, float* scratch /*[kQrWarps][kMaxR]*/,
                             float* out, int op) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int q = 0; q < NV; ++q) {
    if (q >= nv) break;
    float x = v[q];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float y = __shfl_xor_sync(0xffffffffu, x, off);
      x = op == 0 ? x + y : fmaxf(x, y);
    }
    if (lane == 0) scratch[warp * kMaxR + q] = x;
  }
  __syncthreads();
  if (threadIdx.x < nv) {
    float x = scratch[threadIdx.x];
    for (int w = 1; w < kQrWarps; ++w) {
      const float y = scratch[w * kMaxR + threadIdx.x];
      x = op == 0 ? x + y : fmaxf(x, y);
    }
    out[threadIdx.x] = x;
  }
  __syncthreads();
}

template <typename TP>
__device__ __forceinline__ float ldp(const TP* p);
template <>
__device__ __forceinline__ float ldp<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ldp<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

// RT: compile-time bound on r (16, 32 or 64) so per-thread arrays stay in
// registers; columns l >= r are predicated off.
template <int RT, typename TP>
__global__ void __launch_bounds__(kQrThreads) qr_project_kernel(const float* __restrict__ M,
                                                                int p, int r,
                                                                const TP* __restrict__ P,
                                                                float* __restrict__ Vbuf,
                                                                float* __restrict__ Qbuf,
                                                                void* __restrict__ out,
                                                                int hilo) {
  __shared__ float scratch[kQrWarps * kMaxR];
  __shared__ float red[kMaxR];
  __shared__ float vnorm_inv;
  const int i = blockIdx.x;
  const float* m = M + static_cast<size_t>(i) * p * r;
  float* V = Vbuf + static_cast<size_t>(i) * p * r;  // Householder vectors, row-major [p][r]
  float* Q = Qbuf + static_cast<size_t>(i) * p * r;  // thin Q, row-major [p][r]

  // 1. column scaling by 1 / max|M[:, l]|
  {
    float mx[RT];
#pragma unroll
    for (int l = 0; l < RT; ++l) mx[l] = 0.f;
    for (int row = threadIdx.x; row < p; row += kQrThreads) {
#pragma unroll
      for (int l = 0; l < RT; ++l)
        if (l < r) mx[l] = fmaxf(mx[l], fabsf(m[static_cast<size_t>(row) * r + l]));
    }
    block_reduce<RT>(mx, r, scratch, red, 1);
    for (int row = threadIdx.x; row < p; row += kQrThreads) {
#pragma unroll
      for (int l = 0; l < RT; ++l)
        if (l < r) {
          const float sc = red[l] > 0.f ? 1.f / red[l] : 1.f;
          V[static_cast<size_t>(row) * r + l] = m[static_cast<size_t>(row) * r + l] * sc;
        }
    }
    __syncthreads();
  }

  // 2. Householder: for column j, v = x - alpha e_j with alpha = -sign(x_j) ||x||,
  //    normalised; the trailing columns get (I - 2 v v^T).
  for (int j = 0; j < r; ++j) {
    float ss[1] = {0.f};
    for (int row = j + threadIdx.x; row < p; row += kQrThreads) {
      const float x = V[static_cast<size_t>(row) * r + j];
      ss[0] = fmaf(x, x, ss[0]);
    }
    block_reduce<1>(ss, 1, scratch, red, 0);
    if (threadIdx.x == 0) {
      const float norm2 = red[0];
      const float xj = V[static_cast<size_t>(j) * r + j];
      const float alpha = xj >= 0.f ? -sqrtf(norm2) : sqrtf(norm2);
      const float vj = xj - alpha;
      const float vn2 = norm2 - xj * xj + vj * vj;
      V[static_cast<size_t>(j) * r + j] = vj;
      vnorm_inv = vn2 > 0.f ? rsqrtf(vn2) : 0.f;
    }
    __syncthreads();
    const float inv = vnorm_inv;
    for (int row = j + threadIdx.x; row < p; row += kQrThreads)
      V[static_cast<size_t>(row) * r + j] *= inv;
    __syncthreads();
    float dots[RT];
#pragma unroll
    for (int l = 0; l < RT; ++l) dots[l] = 0.f;
    for (int row = j + threadIdx.x; row < p; row += kQrThreads) {
      const float v = V[static_cast<size_t>(row) * r + j];
#pragma unroll
      for (int l = 0; l < RT; ++l)
        if (l > j && l < r) dots[l] = fmaf(v, V[static_cast<size_t>(row) * r + l], dots[l]);
    }
    block_reduce<RT>(dots, r, scratch, red, 0);
    for (int row = j + threadIdx.x; row < p; row += kQrThreads) {
      const float v = V[static_cast<size_t>(row) * r + j];
#pragma unroll
      for (int l = 0; l < RT; ++l)
        if (l > j && l < r) V[static_cast<size_t>(row) * r + l] -= 2.f * v * red[l];
    }
    __syncthreads();
  }

  // 3. Q = H_0 H_1 ... H_{r-1} [I_r; 0], applying the reflectors right to left.
  for (int row = threadIdx.x; row < p; row += kQrThreads)
    for (int l = 0; l < r; ++l) Q[static_cast<size_t>(row) * r + l] = (row == l) ? 1.f : 0.f;
  __syncthreads();
  for (int j = r - 1; j >= 0; --j) {
    float dots[RT];
#pragma unroll
    for (int l = 0; l < RT; ++l) dots[l] = 0.f;
    for (int row = j + threadIdx.x; row < p; row += kQrThreads) {
      const float v = V[static_cast<size_t>(row) * r + j];
#pragma unroll
      for (int l = 0; l < RT; ++l)
        if (l < r) dots[l] = fmaf(v, Q[static_cast<size_t>(row) * r + l], dots[l]);
    }
    block_reduce<RT>(dots, r, scratch, red, 0);
    for (int row = j + threadIdx.x; row < p; row += kQrThreads) {
      const float v = V[static_cast<size_t>(row) * r + j];
#pragma unroll
      for (int l = 0; l < RT; ++l)
        if (l < r) Q[static_cast<size_t>(row) * r + l] -= 2.f * v * red[l];
    }
    __syncthreads();
  }

  // 4. C = Q^T P (r x r), one column b of P at a time; 5. P' = P - Q C.
  //    The reflector store V is reused for P' (no longer needed).
  for (int b = 0; b < r; ++b) {
    float dots[RT];
#pragma unroll
    for (int l = 0; l < RT; ++l) dots[l] = 0.f;
    for (int row = threadIdx.x; row < p; row += kQrThreads) {
      const float pv = ldp(P + static_cast<size_t>(row) * r + b);
#pragma unroll
      for (int a = 0; a < RT; ++a)
        if (a < r) dots[a] = fmaf(Q[static_cast<size_t>(row) * r + a], pv, dots[a]);
    }
    block_reduce<RT>(dots, r, scratch, red, 0);
    for (int row = threadIdx.x; row < p; row += kQrThreads) {
      float v = ldp(P + static_cast<size_t>(row) * r + b);
#pragma unroll
      for (int a = 0; a < RT; ++a)
        if (a < r) v = fmaf(-Q[static_cast<size_t>(row) * r + a], red[a], v);
      V[static_cast<size_t>(row) * r + b] = v;
    }
    __syncthreads();
  }

  // 6. write [Q | P']
  for (int row = threadIdx.x; row < p; row += kQrThreads) {
    if (hilo) {
      __nv_bfloat16* o =
          static_cast<__nv_bfloat16*>(out) + (static_cast<size_t>(i) * p + row) * 4 * r;
      for (int l = 0; l < 2 * r; ++l) {
        const float x = l < r ? Q[static_cast<size_t>(row) * r + l]
                              : V[static_cast<size_t>(row) * r + (l - r)];
        const __nv_bfloat16 hi = __float2bfloat16_rn(x);
        o[l] = hi;
        o[2 * r + l] = __float2bfloat16_rn(x - __bfloat162float(hi));
      }
    } else {
      float* o = static_cast<float*>(out) + (static_cast<size_t>(i) * p + row) * 2 * r;
      for (int l = 0; l < r; ++l) {
        o[l] = Q[static_cast<size_t>(row) * r + l];
        o[r + l] = V[static_cast<size_t>(row) * r + l];
      }
    }
  }
}

template <int RT>
cudaError_t qr_launch(const float* M, int64_t B, int64_t p, int r, const void* P,
                      dprc_dtype pdt, float* V, float* Q, void* out, bool hilo, cudaStream_t s) {
  if (pdt == DPRC_F32)
    qr_project_kernel<RT, float><<<static_cast<unsigned>(B), kQrThreads, 0, s>>>(
        M, static_cast<int>(p), r, static_cast<const float*>(P), V, Q, out, hilo ? 1 : 0);
  else
    qr_project_kernel<RT, __nv_bfloat16><<<static_cast<unsigned>(B), kQrThreads, 0, s>>>(
        M, static_cast<int>(p), r, static_cast<const __nv_bfloat16*>(P), V, Q, out, hilo ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qr_project(const float* M, int64_t B, int64_t p, int r, const void* P,
                              dprc_dtype pdt, float* scratch, void* out, bool hilo,
                              cudaStream_t s) {
  if (r < 1 || r > kMaxR) return cudaErrorInvalidValue;
  // r = 16, p <= 4096: one thread-block cluster per sample
  if (qr_cluster_supported(p, r)) return launch_qr_cluster(M, B, p, P, pdt, out, hilo, s);
  // other r (or p > 4096): one CTA per sample, working copies in global memory
  float* V = scratch;
  float* Q = scratch + static_cast<size_t>(B) * p * r;
  if (r <= 16) return qr_launch<16>(M, B, p, r, P, pdt, V, Q, out, hilo, s);
  if (r <= 32) return qr_launch<32>(M, B, p, r, P, pdt, V, Q, out, hilo, s);
  return qr_launch<64>(M, B, p, r, P, pdt, V, Q, out, hilo, s);
}

}  // namespace dprc
