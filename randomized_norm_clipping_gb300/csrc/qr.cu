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

// ---------------------------------------------------------------------------
// Shared-memory variant (p * r * 4 bytes fit in shared memory): the matrix is
// held column-major in shared memory, each Householder step needs one block
// reduction, and the thin Q is formed in place from the compact WY form
//   H_0 H_1 ... H_{r-1} = I - V T V^T,  T upper triangular,
//   T_jj = 2,  T[0:j, j] = -2 T[0:j, 0:j] (V[:, 0:j]^T v_j)
// (normalised reflectors v_j, H_j = I - 2 v_j v_j^T), so that
//   Q = [I_r; 0] - V (T V_top^T),  V_top = the first r rows of V.
// ---------------------------------------------------------------------------
constexpr int kQrSmemThreads = 512;
constexpr int kQrSmemWarps = kQrSmemThreads / 32;

// Packs two floats into a bf16x2 word (low half first).
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const uint32_t l = __bfloat16_as_ushort(__float2bfloat16_rn(lo));
  const uint32_t h = __bfloat16_as_ushort(__float2bfloat16_rn(hi));
  return l | (h << 16);
}

template <int RT, typename TP>
__global__ void __launch_bounds__(kQrSmemThreads, 1) qr_smem_kernel(const float* __restrict__ M,
                                                                    int p, int r,
                                                                    const TP* __restrict__ P,
                                                                    void* __restrict__ out,
                                                                    int hilo) {
  static_assert(RT == 16, "the row-vector loads and stores assume 16 columns");
  // V: [r][p] fp32 (column l at V + l * p), then P transposed: [r][p] in P's type.
  extern __shared__ float V[];
  TP* PT = reinterpret_cast<TP*>(V + static_cast<size_t>(RT) * p);
  __shared__ float part[kQrSmemWarps][RT];
  __shared__ float coef[RT];
  __shared__ float gram[RT][RT];
  __shared__ float Tm[RT][RT];
  __shared__ float Km[RT][RT];
  __shared__ float Cm[RT][RT];
  __shared__ float inv_s;
  __shared__ float pivot_row[RT];
  const int i = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* m = M + static_cast<size_t>(i) * p * RT;
  constexpr int kRows = 4;  // rows per thread per group in the register-blocked passes
  constexpr int kHhRows = 5;  // rows per thread held through the Householder steps

  // 1. rows of M (and of P) with vector loads, scattered into conflict-free
  //    columns; column maxima on the way.
  float mx[RT];
#pragma unroll
  for (int l = 0; l < RT; ++l) mx[l] = 0.f;
  for (int row = tid; row < p; row += kQrSmemThreads) {
    const float4* src = reinterpret_cast<const float4*>(m + static_cast<size_t>(row) * RT);
    float v[RT];
#pragma unroll
    for (int c4 = 0; c4 < RT / 4; ++c4) {
      const float4 t = src[c4];
      v[4 * c4] = t.x;
      v[4 * c4 + 1] = t.y;
      v[4 * c4 + 2] = t.z;
      v[4 * c4 + 3] = t.w;
    }
#pragma unroll
    for (int l = 0; l < RT; ++l) {
      V[l * p + row] = v[l];
      mx[l] = fmaxf(mx[l], fabsf(v[l]));
      PT[l * p + row] = P[static_cast<size_t>(row) * RT + l];
    }
  }
  //    scale every column by 1 / max |column| (span unchanged)
#pragma unroll
  for (int l = 0; l < RT; ++l) {
    float x = mx[l];
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    if (lane == 0) part[warp][l] = x;
  }
  __syncthreads();
  if (tid < RT) {
    float x = 0.f;
    for (int w = 0; w < kQrSmemWarps; ++w) x = fmaxf(x, part[w][tid]);
    coef[tid] = x > 0.f ? 1.f / x : 1.f;
  }
  __syncthreads();
  for (int row = tid; row < p; row += kQrSmemThreads) {
    float v[RT];
#pragma unroll
    for (int l = 0; l < RT; ++l) v[l] = V[l * p + row];
#pragma unroll
    for (int l = 0; l < RT; ++l) V[l * p + row] = v[l] * coef[l];
  }
  __syncthreads();

  // 2. Householder with the rows in registers: thread t holds rows
  //    t, t + 512, ... (at most kHhRows) for all 16 columns.  Step j needs one
  //    block reduction over rows >= j of
  //      s_l = x . V[:, l],  x = column j,
  //    then every thread applies the reflector to its own rows.  Columns l > j
  //    get (I - 2 v v^T / v^T v); columns l < j already hold the normalised
  //    reflectors v_l, and
  //      v_l^T v_j = (s_l - alpha V[j][l]) / ||v||
  //    is the Gram matrix the compact WY form needs.
  {
    float v[kHhRows][RT];
#pragma unroll
    for (int k = 0; k < kHhRows; ++k) {
      const int row = tid + kQrSmemThreads * k;
#pragma unroll
      for (int l = 0; l < RT; ++l) v[k][l] = row < p ? V[l * p + row] : 0.f;
    }
    for (int j = 0; j < RT; ++j) {
      float sacc[RT];
#pragma unroll
      for (int l = 0; l < RT; ++l) sacc[l] = 0.f;
#pragma unroll
      for (int k = 0; k < kHhRows; ++k) {
        const int row = tid + kQrSmemThreads * k;
        if (row == j) {
#pragma unroll
          for (int l = 0; l < RT; ++l) pivot_row[l] = v[k][l];  // row j, for the pivot
        }
        float xk = 0.f;  // v[k][j], selected without a dynamic register index
#pragma unroll
        for (int l = 0; l < RT; ++l) xk = l == j ? v[k][l] : xk;
        const float xr = (row >= j && row < p) ? xk : 0.f;
#pragma unroll
        for (int l = 0; l < RT; ++l) sacc[l] = fmaf(xr, v[k][l], sacc[l]);
      }
      // butterfly reduce-scatter of the 16 sums over the warp (16 shuffles):
      // afterwards lanes 2c and 2c+1 hold the warp total of sum index idx(c).
      {
        const bool u16 = (lane & 16) != 0;
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          const float mine = u16 ? sacc[t + 8] : sacc[t];
          const float give = u16 ? sacc[t] : sacc[t + 8];
          sacc[t] = mine + __shfl_xor_sync(0xffffffffu, give, 16);
        }
        const bool u8 = (lane & 8) != 0;
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const float mine = u8 ? sacc[t + 4] : sacc[t];
          const float give = u8 ? sacc[t] : sacc[t + 4];
          sacc[t] = mine + __shfl_xor_sync(0xffffffffu, give, 8);
        }
        const bool u4 = (lane & 4) != 0;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float mine = u4 ? sacc[t + 2] : sacc[t];
          const float give = u4 ? sacc[t] : sacc[t + 2];
          sacc[t] = mine + __shfl_xor_sync(0xffffffffu, give, 4);
        }
        const bool u2 = (lane & 2) != 0;
        {
          const float mine = u2 ? sacc[1] : sacc[0];
          const float give = u2 ? sacc[0] : sacc[1];
          sacc[0] = mine + __shfl_xor_sync(0xffffffffu, give, 2);
        }
        sacc[0] += __shfl_xor_sync(0xffffffffu, sacc[0], 1);
        const int idx = (u16 ? 8 : 0) + (u8 ? 4 : 0) + (u4 ? 2 : 0) + (u2 ? 1 : 0);
        if ((lane & 1) == 0) part[warp][idx] = sacc[0];
      }
      __syncthreads();
      if (warp == 0) {
        // lane l < 16 sums column l's partials over the warps, in warp order
        float t = 0.f;
        if (lane < RT)
          for (int w = 0; w < kQrSmemWarps; ++w) t += part[w][lane];
        const float norm2 = __shfl_sync(0xffffffffu, t, j);
        const float xj = pivot_row[j];
        const float nrm = sqrtf(norm2);
        const float alpha = xj >= 0.f ? -nrm : nrm;
        const float vn2 = 2.f * norm2 + 2.f * fabsf(xj) * nrm;  // ||x - alpha e_j||^2
        const float inv = vn2 > 0.f ? rsqrtf(vn2) : 0.f;
        const float vdot = lane < RT ? t - alpha * pivot_row[lane & (RT - 1)] : 0.f;
        if (lane > j && lane < RT) coef[lane] = 2.f * inv * inv * vdot;
        if (lane < j) {
          gram[lane][j] = inv * vdot;
          gram[j][lane] = inv * vdot;
        }
        if (lane == j) {
          coef[j] = alpha;
          gram[j][j] = inv > 0.f ? 1.f : 0.f;
        }
        if (lane == 0) inv_s = inv;
      }
      __syncthreads();
      const float alpha = coef[j], inv = inv_s;
      float cf[RT];
#pragma unroll
      for (int l = 0; l < RT; ++l) cf[l] = l > j ? coef[l] : 0.f;
#pragma unroll
      for (int k = 0; k < kHhRows; ++k) {
        const int row = tid + kQrSmemThreads * k;
        if (row < j || row >= p) continue;
        float xk = 0.f;
#pragma unroll
        for (int l = 0; l < RT; ++l) xk = l == j ? v[k][l] : xk;
        const float vr = row == j ? xk - alpha : xk;
        // columns l > j get the reflector; column j becomes the normalised v_j
#pragma unroll
        for (int l = 0; l < RT; ++l)
          v[k][l] = l > j ? fmaf(-cf[l], vr, v[k][l]) : (l == j ? vr * inv : v[k][l]);
      }
    }
#pragma unroll
    for (int k = 0; k < kHhRows; ++k) {
      const int row = tid + kQrSmemThreads * k;
      if (row < p)
#pragma unroll
        for (int l = 0; l < RT; ++l) V[l * p + row] = v[k][l];
    }
    __syncthreads();
  }

  // T (upper triangular), column by column: lane a of warp 0 computes T[a][j]
  if (warp == 0) {
    for (int j = 0; j < RT; ++j) {
      float t = 0.f;
      if (lane < j)
        for (int b = lane; b < j; ++b) t = fmaf(Tm[lane][b], gram[b][j], t);
      __syncwarp();
      if (lane < j) Tm[lane][j] = -2.f * t;
      if (lane == j) Tm[j][j] = 2.f;
      if (lane > j && lane < RT) Tm[lane][j] = 0.f;
      __syncwarp();
    }
  }
  __syncthreads();
  // K = T V_top^T: K[a][l] = sum_{a <= b <= l} T[a][b] (reflector b at row l)
  for (int e = tid; e < RT * RT; e += kQrSmemThreads) {
    const int a = e / RT, l = e % RT;
    float t = 0.f;
    for (int b = a; b <= l; ++b) t = fmaf(Tm[a][b], V[b * p + l], t);
    Km[a][l] = t;
  }
  __syncthreads();

  // 4. Q = [I_r; 0] - V K, in place.  Rows go in groups: each thread holds
  //    kRows rows in registers and walks a, reusing K's row a.  A row only
  //    reads its own reflector entries, so writing it back in place is safe.
  for (int g0 = 0; g0 < p; g0 += kQrSmemThreads * kRows) {
    float q[kRows][RT];
#pragma unroll
    for (int k = 0; k < kRows; ++k)
#pragma unroll
      for (int l = 0; l < RT; ++l) q[k][l] = (g0 + tid + kQrSmemThreads * k == l) ? 1.f : 0.f;
    for (int a = 0; a < RT; ++a) {
      float krow[RT];
#pragma unroll
      for (int l = 0; l < RT; ++l) krow[l] = Km[a][l];
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        const int row = g0 + tid + kQrSmemThreads * k;
        const float va = (row < p && row >= a) ? V[a * p + row] : 0.f;
#pragma unroll
        for (int l = 0; l < RT; ++l) q[k][l] = fmaf(-va, krow[l], q[k][l]);
      }
    }
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      const int row = g0 + tid + kQrSmemThreads * k;
      if (row < p)
#pragma unroll
        for (int l = 0; l < RT; ++l) V[l * p + row] = q[k][l];
    }
  }
  __syncthreads();

  // 5. C = Q^T P (16 x 16): warp w owns the 4 x 4 block (a0, b0); lane walks
  //    rows lane, lane + 32, ... (conflict-free column reads), then a warp
  //    reduction of the 16 sums.
  {
    const int a0 = (warp >> 2) * 4, b0 = (warp & 3) * 4;
    float c[4][4];
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) c[x][y] = 0.f;
    for (int row = lane; row < p; row += 32) {
      float qa[4], pb[4];
#pragma unroll
      for (int x = 0; x < 4; ++x) qa[x] = V[(a0 + x) * p + row];
#pragma unroll
      for (int y = 0; y < 4; ++y) pb[y] = ldp(PT + (b0 + y) * p + row);
#pragma unroll
      for (int x = 0; x < 4; ++x)
#pragma unroll
        for (int y = 0; y < 4; ++y) c[x][y] = fmaf(qa[x], pb[y], c[x][y]);
    }
#pragma unroll
    for (int x = 0; x < 4; ++x)
#pragma unroll
      for (int y = 0; y < 4; ++y) {
        float t = c[x][y];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
        if (lane == 0) Cm[a0 + x][b0 + y] = t;
      }
  }
  __syncthreads();

  // 6. P' = P - Q C (same blocking as step 4); each thread writes whole rows
  //    of [Q | P'] with 16-byte stores.
  for (int g0 = 0; g0 < p; g0 += kQrSmemThreads * kRows) {
    float pp[kRows][RT];
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      const int row = g0 + tid + kQrSmemThreads * k;
#pragma unroll
      for (int l = 0; l < RT; ++l) pp[k][l] = row < p ? ldp(PT + l * p + row) : 0.f;
    }
    for (int a = 0; a < RT; ++a) {
      float crow[RT];
#pragma unroll
      for (int l = 0; l < RT; ++l) crow[l] = Cm[a][l];
#pragma unroll
      for (int k = 0; k < kRows; ++k) {
        const int row = g0 + tid + kQrSmemThreads * k;
        const float qa = row < p ? V[a * p + row] : 0.f;
#pragma unroll
        for (int l = 0; l < RT; ++l) pp[k][l] = fmaf(-qa, crow[l], pp[k][l]);
      }
    }
#pragma unroll
    for (int k = 0; k < kRows; ++k) {
      const int row = g0 + tid + kQrSmemThreads * k;
      if (row >= p) continue;
      float qv[RT];
#pragma unroll
      for (int l = 0; l < RT; ++l) qv[l] = V[l * p + row];
      if (hilo) {
        // [Q_hi | P'_hi | Q_lo | P'_lo], 16 bf16 each = 2 x 16 B each
        uint32_t w[32];
#pragma unroll
        for (int l = 0; l < RT; l += 2) {
          const float q0h = __bfloat162float(__float2bfloat16_rn(qv[l]));
          const float q1h = __bfloat162float(__float2bfloat16_rn(qv[l + 1]));
          const float p0h = __bfloat162float(__float2bfloat16_rn(pp[k][l]));
          const float p1h = __bfloat162float(__float2bfloat16_rn(pp[k][l + 1]));
          w[l / 2] = pack_bf16x2(qv[l], qv[l + 1]);
          w[8 + l / 2] = pack_bf16x2(pp[k][l], pp[k][l + 1]);
          w[16 + l / 2] = pack_bf16x2(qv[l] - q0h, qv[l + 1] - q1h);
          w[24 + l / 2] = pack_bf16x2(pp[k][l] - p0h, pp[k][l + 1] - p1h);
        }
        uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) +
                                            (static_cast<size_t>(i) * p + row) * 4 * RT);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4)
          o[c4] = make_uint4(w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
      } else {
        float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) +
                                              (static_cast<size_t>(i) * p + row) * 2 * RT);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          o[c4] = make_float4(qv[4 * c4], qv[4 * c4 + 1], qv[4 * c4 + 2], qv[4 * c4 + 3]);
#pragma unroll
        for (int c4 = 0; c4 < 4; ++c4)
          o[4 + c4] = make_float4(pp[k][4 * c4], pp[k][4 * c4 + 1], pp[k][4 * c4 + 2],
                                  pp[k][4 * c4 + 3]);
      }
    }
  }
}

template <int RT>
cudaError_t qr_smem_launch(const float* M, int64_t B, int64_t p, int r, const void* P,
                           dprc_dtype pdt, void* out, bool hilo, cudaStream_t s) {
  const int smem = static_cast<int>(p * RT * (sizeof(float) + (pdt == DPRC_F32 ? 4 : 2)));
  if (pdt == DPRC_F32) {
    auto k = qr_smem_kernel<RT, float>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k<<<static_cast<unsigned>(B), kQrSmemThreads, smem, s>>>(M, static_cast<int>(p), r,
                                                            static_cast<const float*>(P), out,
                                                            hilo ? 1 : 0);
  } else {
    auto k = qr_smem_kernel<RT, __nv_bfloat16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    k<<<static_cast<unsigned>(B), kQrSmemThreads, smem, s>>>(
        M, static_cast<int>(p), r, static_cast<const __nv_bfloat16*>(P), out, hilo ? 1 : 0);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_qr_project(const float* M, int64_t B, int64_t p, int r, const void* P,
                              dprc_dtype pdt, float* scratch, void* out, bool hilo,
                              cudaStream_t s) {
  if (r < 1 || r > kMaxR) return cudaErrorInvalidValue;
  // r = 16, p <= 4096: one thread-block cluster per sample
  if (qr_cluster_supported(p, r)) return launch_qr_cluster(M, B, p, P, pdt, out, hilo, s);
  // shared-memory variant for r = 16 when M (fp32) and P^T fit: p <= 2260
  // with bf16 P, p <= 1696 with fp32 P
  if (r == 16 && p <= 5 * kQrSmemThreads && p * 16 * (4 + (pdt == DPRC_F32 ? 4 : 2)) <= 212 * 1024)
    return qr_smem_launch<16>(M, B, p, r, P, pdt, out, hilo, s);
  float* V = scratch;
  float* Q = scratch + static_cast<size_t>(B) * p * r;
  if (r <= 16) return qr_launch<16>(M, B, p, r, P, pdt, V, Q, out, hilo, s);
  if (r <= 32) return qr_launch<32>(M, B, p, r, P, pdt, V, Q, out, hilo, s);
  return qr_launch<64>(M, B, p, r, P, pdt, V, Q, out, hilo, s);
}

}  // namespace dprc
