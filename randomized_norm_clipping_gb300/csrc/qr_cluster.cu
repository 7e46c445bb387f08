// Hutch++ middle step on a thread-block cluster per sample (papernotes.org,
// "Key design > Hutch++ head-tail decomposition": Q is an orthonormal basis of
// Col(O S); the tail runs Hutchinson on the residual (I - Q Q^T)):
//
//   Q_i  = thin Q of a Householder QR of M_i = O_i S      (p x 16, per sample)
//   P'_i = P - Q_i (Q_i^T P)
//
// written as [Q_i | P'_i] (bf16 hi/lo planes or fp32) for the next sketch.
//
// The QR is a chain of 16 dependent reductions over the p rows, so one CTA per
// sample leaves the GPU nearly idle.  Here the p rows of a sample are spread
// over a cluster of 8 CTAs x 256 threads (one or two rows per thread, held in
// registers for the whole factorisation); each Householder step is one
// all-reduce across the cluster through distributed shared memory:
//
//   every CTA reduces its rows' 16 dot products s_l = x . V[:, l] (a warp
//   butterfly, then the warps in order), warp 0 stores them, together with the
//   pivot row (held by rank 0, zeros elsewhere), into a slot of every CTA of
//   the cluster with asynchronous stores counted on that CTA's barrier; each
//   CTA then sums the 8 slots in rank order, so every CTA holds the same
//   totals and applies the reflector to its own rows.
//
// The same exchange serves the column scaling before the steps and the
// 16 x 16 product C = Q^T P after them.  Every CTA rebuilds, from the
// exchanged values, the Gram matrix of the reflectors, the top 16 rows of V
// and the compact-WY factor T, so Q = E - V (T V_top^T) and P' need no
// further exchange.  Sums run in a fixed order (deterministic).
//
// With `rc` set, rank 0 of each cluster also writes the sample's factors for
// a caller that forms X Q as (X M) R^-1: R of the scaled M (its rows fall out
// of the step totals), the column scales and C.  The kernel lets the next
// kernel in the stream start at once (programmatic dependent launch); that
// one must not read what this kernel writes before it completes.
//
// Householder QR stays orthonormal when M is rank deficient (a zero reflector
// is the identity), which is exactly the low-rank case where Hutch++ is exact;
// the columns are first scaled by their largest magnitude (span unchanged).

#include <cuda_bf16.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace dprc {
namespace {

constexpr int kR = 16;       // columns (r)
constexpr int kCl = 8;       // CTAs per sample
constexpr int kCt = 256;     // threads per CTA
constexpr int kCw = kCt / 32;
constexpr int kE = kR * kR;  // entries of a 16 x 16 matrix
constexpr int kEpt = kCt >= kE ? 1 : kE / kCt;       // of them per thread
constexpr int kCrows = kR / kCw > 0 ? kR / kCw : 1;  // rows of C = Q^T P per warp
static_assert((kCt >= kE || kE % kCt == 0) && (kR % kCw == 0 || kCw % kR == 0), "CTA size");
constexpr int kXch = 256;    // floats per rank slot of the exchange buffer
constexpr int kRC = 2 * kE + kR;  // factors per sample: R (row-major), column scales, C

template <typename TP>
__device__ __forceinline__ float ld_elem(const TP* p);
template <>
__device__ __forceinline__ float ld_elem<float>(const float* p) { return *p; }
template <>
__device__ __forceinline__ float ld_elem<__nv_bfloat16>(const __nv_bfloat16* p) {
  return __bfloat162float(*p);
}

__device__ __forceinline__ uint32_t pack2(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Butterfly reduce-scatter of 16 per-lane values (sum or max) across the
// warp: afterwards lanes 2c and 2c+1 hold the warp total of index idx(lane).
template <bool kMax>
__device__ __forceinline__ float warp_scatter16(float (&v)[16], int lane, int& idx) {
  auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
  const bool u16 = (lane & 16) != 0;
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const float mine = u16 ? v[t + 8] : v[t];
    const float give = u16 ? v[t] : v[t + 8];
    v[t] = op(mine, __shfl_xor_sync(0xffffffffu, give, 16));
  }
  const bool u8 = (lane & 8) != 0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const float mine = u8 ? v[t + 4] : v[t];
    const float give = u8 ? v[t] : v[t + 4];
    v[t] = op(mine, __shfl_xor_sync(0xffffffffu, give, 8));
  }
  const bool u4 = (lane & 4) != 0;
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const float mine = u4 ? v[t + 2] : v[t];
    const float give = u4 ? v[t] : v[t + 2];
    v[t] = op(mine, __shfl_xor_sync(0xffffffffu, give, 4));
  }
  const bool u2 = (lane & 2) != 0;
  {
    const float mine = u2 ? v[1] : v[0];
    const float give = u2 ? v[0] : v[1];
    v[0] = op(mine, __shfl_xor_sync(0xffffffffu, give, 2));
  }
  v[0] = op(v[0], __shfl_xor_sync(0xffffffffu, v[0], 1));
  idx = (u16 ? 8 : 0) + (u8 ? 4 : 0) + (u4 ? 2 : 0) + (u2 ? 1 : 0);
  return v[0];
}

struct Exchange {
  float (*buf)[kCl][kXch];  // [2][kCl][kXch]
  uint64_t* bar;            // [2]
  int rank;
};

// Round `rnd` of the cluster all-gather, called by warp 0 once this CTA's
// `n` values (a multiple of 4) sit in the local buffer slot [rnd & 1][rank]:
// lane 0 announces the (kCl - 1) n floats this CTA will receive (the one
// arrival the barrier counts; it also publishes the local slot), and lane
// r < kCl, r != rank, copies the slot into the same slot of CTA r with
// asynchronous 16-byte stores that complete on that CTA's barrier.  A peer can
// be at most one round ahead (it needs this CTA's data of the current round
// first), so two buffers and two barriers suffice.
__device__ __forceinline__ void xch_send(const Exchange& x, int rnd, int n, int lane) {
  const int b = rnd & 1;
  __syncwarp();
  if (lane == 0) mbar_arrive_expect_tx(&x.bar[b], static_cast<uint32_t>((kCl - 1) * n * 4));
  if (lane < kCl && lane != x.rank) {
    const float4* src = reinterpret_cast<const float4*>(&x.buf[b][x.rank][0]);
    const uint32_t dst = map_to_rank(&x.buf[b][x.rank][0], lane);
    const uint32_t rbar = map_to_rank(&x.bar[b], lane);
    for (int q = 0; q < n / 4; ++q) st_async_f4(dst + 16 * q, src[q], rbar);
  }
}

// Every thread: wait until all CTAs' slots of round `rnd` have arrived.
__device__ __forceinline__ bool xch_wait(const Exchange& x, int rnd) {
  return mbar_wait(&x.bar[rnd & 1], static_cast<uint32_t>(rnd >> 1) & 1, DPRC_DEVERR_CLUSTER);
}

template <int RPT, typename TP>
__global__ void __launch_bounds__(kCt, 1)
    qr_cluster_kernel(const float* __restrict__ M, int p, const TP* __restrict__ P,
                      void* __restrict__ out, int hilo, float* __restrict__ rc) {
  __shared__ float xbuf[2][kCl][kXch];
  __shared__ __align__(8) uint64_t xbar[2];
  __shared__ float part[kCw][kR];
  __shared__ float piv[kR];
  __shared__ float gram[kR][kR];
  __shared__ float vtop[kR][kR];
  __shared__ float Tm[kR][kR];
  __shared__ float Km[kR][kR];
  __shared__ float Cm[kR * kR];
  __shared__ float Rsm[kR][kR];  // R of the scaled M
  __shared__ float scm[kR];      // column scales
  __shared__ float cpart[kCw][kE];  // per-warp parts of this CTA's part of C

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // Each sample's rows are spread over one cluster of kCl CTAs; a launch of
  // any other cluster shape would address ranks that do not exist: refuse it.
  if (cluster_nctarank() != static_cast<uint32_t>(kCl)) {
    if (tid == 0) record_error(DPRC_DEVERR_LAUNCH);
    return;
  }
  pdl_launch_dependents();  // the next kernel reads nothing this one writes before it ends
  const int rank = static_cast<int>(cluster_ctarank());
  const int i = blockIdx.x / kCl;
  const float* m_i = M + static_cast<size_t>(i) * p * kR;
  Exchange x;
  x.buf = xbuf;
  x.bar = xbar;
  x.rank = rank;
  bool ok = true;

  if (tid == 0) {
    mbar_init(&xbar[0], 1);
    mbar_init(&xbar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  cluster_sync_all();  // every CTA's barriers exist before the first remote arrive

  // rows of this thread: k * (kCl * kCt) + rank * kCt + tid (rank 0 holds rows 0..kCt-1)
  auto row_of = [&](int k) { return k * (kCl * kCt) + rank * kCt + tid; };
  float v[RPT][kR];
#pragma unroll
  for (int k = 0; k < RPT; ++k) {
    const int row = row_of(k);
    if (row < p) {
      const float4* src = reinterpret_cast<const float4*>(m_i + static_cast<size_t>(row) * kR);
#pragma unroll
      for (int c4 = 0; c4 < kR / 4; ++c4) {
        const float4 t = src[c4];
        v[k][4 * c4] = t.x;
        v[k][4 * c4 + 1] = t.y;
        v[k][4 * c4 + 2] = t.z;
        v[k][4 * c4 + 3] = t.w;
      }
    } else {
#pragma unroll
      for (int l = 0; l < kR; ++l) v[k][l] = 0.f;
    }
  }

  // ---- round 0: column maxima; scale columns by 1 / max |column| ----
  {
    float mx[kR];
#pragma unroll
    for (int l = 0; l < kR; ++l) {
      float t = 0.f;
#pragma unroll
      for (int k = 0; k < RPT; ++k) t = fmaxf(t, fabsf(v[k][l]));
      mx[l] = t;
    }
    int idx;
    const float w = warp_scatter16<true>(mx, lane, idx);
    if ((lane & 1) == 0) part[warp][idx] = w;
    __syncthreads();
    if (warp == 0) {
      float t = 0.f;
      if (lane < kR)
        for (int ww = 0; ww < kCw; ++ww) t = fmaxf(t, part[ww][lane]);
      xbuf[0][rank][lane] = t;
      xch_send(x, 0, 32, lane);
    }
    if (!xch_wait(x, 0)) ok = false;
    float tot = 0.f;
    if (lane < kR)
      for (int r = 0; r < kCl; ++r) tot = fmaxf(tot, xbuf[0][r][lane]);
    const float sc = tot > 0.f ? 1.f / tot : 1.f;
    if (warp == 0 && lane < kR) scm[lane] = sc;
#pragma unroll
    for (int l = 0; l < kR; ++l) {
      const float s_l = __shfl_sync(0xffffffffu, sc, l);
#pragma unroll
      for (int k = 0; k < RPT; ++k) v[k][l] *= s_l;
    }
  }

  // ---- rounds 1..16: Householder steps ----
  for (int j = 0; j < kR; ++j) {
    const int rnd = 1 + j;
    float sacc[kR];
#pragma unroll
    for (int l = 0; l < kR; ++l) sacc[l] = 0.f;
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      const int row = row_of(k);
      float xk = 0.f;  // v[k][j] without a dynamic register index
#pragma unroll
      for (int l = 0; l < kR; ++l) xk = l == j ? v[k][l] : xk;
      if (row == j) {
#pragma unroll
        for (int l = 0; l < kR; ++l) piv[l] = v[k][l];
      }
      const float xr = (row >= j && row < p) ? xk : 0.f;
#pragma unroll
      for (int l = 0; l < kR; ++l) sacc[l] = fmaf(xr, v[k][l], sacc[l]);
    }
    int idx;
    const float w = warp_scatter16<false>(sacc, lane, idx);
    if ((lane & 1) == 0) part[warp][idx] = w;
    __syncthreads();
    if (warp == 0) {
      // lanes 0..15: this CTA's s_l (warps in order); lanes 16..31: the pivot
      // row (rank 0 holds it; the others send zeros)
      float t = 0.f;
      if (lane < kR) {
        for (int ww = 0; ww < kCw; ++ww) t += part[ww][lane];
      } else if (rank == 0) {
        t = piv[lane - kR];
      }
      xbuf[rnd & 1][rank][lane] = t;
      xch_send(x, rnd, 32, lane);
    }
    if (!xch_wait(x, rnd)) ok = false;
    // every warp: lane l < 16 -> s_l, lane 16 + l -> pivot row entry l
    float tot = 0.f;
    for (int r = 0; r < kCl; ++r) tot += xbuf[rnd & 1][r][lane];
    const float norm2 = __shfl_sync(0xffffffffu, tot, j);
    const float xj = __shfl_sync(0xffffffffu, tot, kR + j);
    const float pv = __shfl_sync(0xffffffffu, tot, kR + (lane & (kR - 1)));
    const float nrm = sqrtf(norm2);
    const float alpha = xj >= 0.f ? -nrm : nrm;
    const float vn2 = 2.f * norm2 + 2.f * fabsf(xj) * nrm;  // ||x - alpha e_j||^2
    const float inv = vn2 > 0.f ? rsqrtf(vn2) : 0.f;
    const float vdot = tot - alpha * pv;  // lanes < 16: v_j . column l
    const float cf_lane = lane > j && lane < kR ? 2.f * inv * inv * vdot : 0.f;
    if (warp == 0 && lane < kR) {
      if (lane < j) {
        gram[lane][j] = inv * vdot;
        gram[j][lane] = inv * vdot;
        vtop[j][lane] = pv;  // reflector `lane` at row j
      } else if (lane == j) {
        gram[j][j] = inv > 0.f ? 1.f : 0.f;
        vtop[j][j] = (xj - alpha) * inv;
      } else {
        vtop[j][lane] = 0.f;
      }
      // row j of R: alpha on the diagonal, the pivot row after the reflector right of it
      Rsm[j][lane] = lane < j ? 0.f : (lane == j ? alpha : fmaf(-cf_lane, xj - alpha, pv));
    }
    float cf[kR];
#pragma unroll
    for (int l = 0; l < kR; ++l) cf[l] = __shfl_sync(0xffffffffu, cf_lane, l);
#pragma unroll
    for (int k = 0; k < RPT; ++k) {
      const int row = row_of(k);
      if (row < j || row >= p) continue;
      float xk = 0.f;
#pragma unroll
      for (int l = 0; l < kR; ++l) xk = l == j ? v[k][l] : xk;
      const float vr = row == j ? xk - alpha : xk;
      // columns l > j get the reflector; column j becomes the normalised v_j
#pragma unroll
      for (int l = 0; l < kR; ++l)
        v[k][l] = l > j ? fmaf(-cf[l], vr, v[k][l]) : (l == j ? vr * inv : v[k][l]);
    }
  }
  __syncthreads();  // gram and vtop complete

  // T of the compact WY form Q = E - V T V^T E.  For normalised reflectors
  // T^-1 = I/2 + N, N the strictly upper part of their Gram matrix, so with
  // X = 2N (nilpotent, X^16 = 0)
  //   T = 2 (I + X)^-1 = 2 (I - X)(I + X^2)(I + X^4)(I + X^8):
  // six 16 x 16 products, one entry per thread.  Then K = T V_top^T.
  {
    // entries e = tid + kCt m (m < kEpt) of each 16 x 16 matrix; threads
    // beyond the 256 entries only keep step
    const bool ent = tid < kE;
    float* X = &Tm[0][0];   // X, then its powers
    float* Y = &Km[0][0];   // running product
#pragma unroll
    for (int m = 0; m < kEpt; ++m) {
      const int e = tid + kCt * m, a = (e >> 4) & (kR - 1), l = e & 15;
      if (ent) {
        X[e] = l > a ? 2.f * gram[a][l] : 0.f;
        Y[e] = (l == a ? 1.f : 0.f) - (l > a ? 2.f * gram[a][l] : 0.f);  // I - X
      }
    }
    __syncthreads();
    for (int sq = 0; sq < 3; ++sq) {
      // X <- X^2 (X^2, X^4, X^8), then Y <- Y (I + X)
      float t[kEpt];
#pragma unroll
      for (int m = 0; m < kEpt; ++m) {
        const int e = tid + kCt * m, a = (e >> 4) & (kR - 1), l = e & 15;
        t[m] = 0.f;
#pragma unroll
        for (int b = 0; b < kR; ++b) t[m] = fmaf(X[a * kR + b], X[b * kR + l], t[m]);
      }
      __syncthreads();
#pragma unroll
      for (int m = 0; m < kEpt; ++m)
        if (ent) X[tid + kCt * m] = t[m];
      __syncthreads();
#pragma unroll
      for (int m = 0; m < kEpt; ++m) {
        const int e = tid + kCt * m, a = (e >> 4) & (kR - 1), l = e & 15;
        t[m] = Y[a * kR + l];
#pragma unroll
        for (int b = 0; b < kR; ++b) t[m] = fmaf(Y[a * kR + b], X[b * kR + l], t[m]);
      }
      __syncthreads();
#pragma unroll
      for (int m = 0; m < kEpt; ++m)
        if (ent) Y[tid + kCt * m] = t[m];
      __syncthreads();
    }
    // T = 2 Y (upper triangular); K[a][l] = sum_{a <= b <= l} T[a][b] V_top[l][b]
    float t[kEpt];
#pragma unroll
    for (int m = 0; m < kEpt; ++m) {
      const int e = tid + kCt * m, a = (e >> 4) & (kR - 1), l = e & 15;
      t[m] = 0.f;
      for (int b = a; b <= l; ++b) t[m] = fmaf(2.f * Y[a * kR + b], vtop[l][b], t[m]);
    }
    __syncthreads();
#pragma unroll
    for (int m = 0; m < kEpt; ++m)
      if (ent) (&Km[0][0])[tid + kCt * m] = t[m];
  }
  __syncthreads();

  // this thread's rows of P; its rows of Q = [I; 0] - V K are formed from V
  // and K when needed (entry a of row `row`: [row == a] - sum over the
  // reflectors b <= row of v_b K[b][a])
  float pk[RPT][kR];
#pragma unroll
  for (int k = 0; k < RPT; ++k) {
    const int row = row_of(k);
#pragma unroll
    for (int l = 0; l < kR; ++l)
      pk[k][l] = row < p ? ld_elem(P + static_cast<size_t>(row) * kR + l) : 0.f;
  }
  auto q_entry = [&](int k, int a) {
    const int row = row_of(k);
    float q = row == a ? 1.f : 0.f;
#pragma unroll
    for (int b = 0; b < kR; ++b) {
      const float vb = (row < p && row >= b) ? v[k][b] : 0.f;
      q = fmaf(-vb, Km[b][a], q);
    }
    return row < p ? q : 0.f;
  };

  // this CTA's part of C = Q^T P: for each row a of C the warp reduce-scatters
  // its rows' products q_a p_l (lanes 2c, 2c+1 then hold the warp's total of
  // one column), and the warps' totals are added in warp order
#pragma unroll 1
  for (int a = 0; a < kR; ++a) {
    float qa[RPT];
#pragma unroll
    for (int k = 0; k < RPT; ++k) qa[k] = q_entry(k, a);
    float c[kR];
#pragma unroll
    for (int l = 0; l < kR; ++l) {
      c[l] = 0.f;
#pragma unroll
      for (int k = 0; k < RPT; ++k) c[l] = fmaf(qa[k], pk[k][l], c[l]);
    }
    int idx;
    const float w = warp_scatter16<false>(c, lane, idx);
    if ((lane & 1) == 0) cpart[warp][a * kR + idx] = w;
  }
  __syncthreads();
#pragma unroll
  for (int m = 0; m < kEpt; ++m)
    if (tid + kCt * m < kE) {
      float t = 0.f;
#pragma unroll
      for (int w2 = 0; w2 < kCw; ++w2) t += cpart[w2][tid + kCt * m];
      Cm[tid + kCt * m] = t;
    }
  __syncthreads();
  // round 17: all-gather the 256 partials; every thread sums its entries
#pragma unroll
  for (int m = 0; m < kEpt; ++m)
    if (tid < kE) xbuf[(1 + kR) & 1][rank][tid + kCt * m] = Cm[tid + kCt * m];
  __syncthreads();
  if (warp == 0) xch_send(x, 1 + kR, kE, lane);
  if (!xch_wait(x, 1 + kR)) ok = false;
  {
    float t[kEpt];
#pragma unroll
    for (int m = 0; m < kEpt; ++m) {
      t[m] = 0.f;
      if (tid < kE)
        for (int r = 0; r < kCl; ++r) t[m] += xbuf[(1 + kR) & 1][r][tid + kCt * m];
    }
    __syncthreads();  // everyone has read this CTA's partial of Cm
#pragma unroll
    for (int m = 0; m < kEpt; ++m)
      if (tid < kE) Cm[tid + kCt * m] = t[m];
  }
  __syncthreads();
  if (rc != nullptr && rank == 0 && ok) {
    float* f = rc + static_cast<size_t>(i) * kRC;
#pragma unroll
    for (int m = 0; m < kEpt; ++m)
      if (tid < kE) {
        f[tid + kCt * m] = (&Rsm[0][0])[tid + kCt * m];
        f[kE + kR + tid + kCt * m] = Cm[tid + kCt * m];
      }
    if (tid < kR) f[kE + tid] = scm[tid];
  }

  // P' = P - Q C and the output rows
#pragma unroll
  for (int k = 0; k < RPT; ++k) {
    const int row = row_of(k);
    if (row >= p || out == nullptr) continue;
    float q[kR], pp[kR];
#pragma unroll
    for (int l = 0; l < kR; ++l) {
      q[l] = q_entry(k, l);
      pp[l] = pk[k][l];
    }
#pragma unroll
    for (int a = 0; a < kR; ++a)
#pragma unroll
      for (int l = 0; l < kR; ++l) pp[l] = fmaf(-q[a], Cm[a * kR + l], pp[l]);
    if (!ok) continue;
    if (hilo) {
      // [Q_hi | P'_hi | Q_lo | P'_lo], 16 bf16 each
      uint32_t w[32];
#pragma unroll
      for (int l = 0; l < kR; l += 2) {
        const float q0h = __bfloat162float(__float2bfloat16_rn(q[l]));
        const float q1h = __bfloat162float(__float2bfloat16_rn(q[l + 1]));
        const float p0h = __bfloat162float(__float2bfloat16_rn(pp[l]));
        const float p1h = __bfloat162float(__float2bfloat16_rn(pp[l + 1]));
        w[l / 2] = pack2(q[l], q[l + 1]);
        w[8 + l / 2] = pack2(pp[l], pp[l + 1]);
        w[16 + l / 2] = pack2(q[l] - q0h, q[l + 1] - q1h);
        w[24 + l / 2] = pack2(pp[l] - p0h, pp[l + 1] - p1h);
      }
      uint4* o = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(out) +
                                          (static_cast<size_t>(i) * p + row) * 4 * kR);
#pragma unroll
      for (int c4 = 0; c4 < 8; ++c4)
        o[c4] = make_uint4(w[4 * c4], w[4 * c4 + 1], w[4 * c4 + 2], w[4 * c4 + 3]);
    } else {
      float4* o = reinterpret_cast<float4*>(static_cast<float*>(out) +
                                            (static_cast<size_t>(i) * p + row) * 2 * kR);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
        o[c4] = make_float4(q[4 * c4], q[4 * c4 + 1], q[4 * c4 + 2], q[4 * c4 + 3]);
#pragma unroll
      for (int c4 = 0; c4 < 4; ++c4)
        o[4 + c4] = make_float4(pp[4 * c4], pp[4 * c4 + 1], pp[4 * c4 + 2], pp[4 * c4 + 3]);
    }
  }
  cluster_sync_all();  // no CTA leaves while a peer may still address its shared memory
}

template <int RPT, typename TP>
cudaError_t launch_rpt(const float* M, int64_t B, int64_t p, const void* P, void* out, bool hilo,
                       float* rc, cudaStream_t s) {
  auto kern = qr_cluster_kernel<RPT, TP>;
  constexpr int kMaxDev = 64;
  static std::atomic<int> done[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev || !done[dev].load(std::memory_order_acquire)) {
    // an SM that takes a QR CTA (about 31 KB of shared memory) keeps its
    // largest shared-memory carve-out, so two CTAs of the sketch or the
    // projection of the pass that runs beside the QR fit next to it
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                             cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (kCl > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    if (dev >= 0 && dev < kMaxDev) done[dev].store(1, std::memory_order_release);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B * kCl));
  cfg.blockDim = dim3(kCt);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = kCl;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, M, static_cast<int>(p), static_cast<const TP*>(P), out,
                            hilo ? 1 : 0, rc);
}

template <int RPT>
cudaError_t launch_dt(const float* M, int64_t B, int64_t p, const void* P, dprc_dtype pdt,
                      void* out, bool hilo, float* rc, cudaStream_t s) {
  return pdt == DPRC_F32 ? launch_rpt<RPT, float>(M, B, p, P, out, hilo, rc, s)
                         : launch_rpt<RPT, __nv_bfloat16>(M, B, p, P, out, hilo, rc, s);
}

}  // namespace

cudaError_t read_device_error_qr(int32_t* out, bool reset) {
  return read_tu_device_error(out, reset);
}

bool qr_cluster_supported(int64_t p, int r) { return r == kR && p >= kR && p <= 2 * kCl * kCt; }

int qr_factor_floats() { return kRC; }

cudaError_t launch_qr_cluster(const float* M, int64_t B, int64_t p, const void* P, dprc_dtype pdt,
                              void* out, bool hilo, cudaStream_t s, float* rc) {
  if (p <= kCl * kCt) return launch_dt<1>(M, B, p, P, pdt, out, hilo, rc, s);
  return launch_dt<2>(M, B, p, P, pdt, out, hilo, rc, s);
}

}  // namespace dprc
