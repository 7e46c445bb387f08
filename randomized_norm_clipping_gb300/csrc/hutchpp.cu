// Hutch++ on tensor cores with the QR beside the third pass ("Efficient
// DP-SGD for LLMs with Randomized Clipping", papernotes.org, "Key design >
// Hutch++ head-tail decomposition": Q an orthonormal basis of Col(O S), the
// head ||X Q||_F^2 taken exactly, the tail a Hutchinson estimate on the
// residual (I - Q Q^T) with weight 1/r; X = A_i^T G_i, O = X^T X).
//
// The third pass needs X Q and X P' with P' = P - Q C, C = Q^T P.  For M of
// full column rank, Q = M diag(s) R^-1 (M diag(s) = Q R, the QR of the
// column-scaled M), so
//
//   X Q  = (X M) diag(s) R^-1,        X P' = X P - (X Q) C,
//
// and the pass can stream X M while the QR runs: X P comes with the first
// pass (its sketch operand is [S | P], packed here), X M with the third, and
// the third pass's projection epilogue applies the small factors row by row
// (tc_proj.cu, mode kColprojHpp).
//
// The solve divides by the diagonal of R, so it magnifies the rounding of the
// bf16 hi/lo sketches (relative 2^-17) in X M by |R_jj|^-1 relative to the
// column's norm.  A column j with |R_jj| at most kHppDropTau = 1e-3 of its
// column norm is left out of X Q (set to zero; the head and the tail then
// both leave q_j out): M is numerically rank deficient there, q_j lies in the
// part of Col(O S) that rounding decides, and X q_j carries a share of n of
// the order of that ratio.  Leaving it out and keeping it amplified err in
// opposite directions; 1e-3 sits between them (about the square root of the
// sketch's relative rounding), and on the benchmark batch and the test
// shapes the result stays within 2e-4 of the Householder-Q estimate.

#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace dprc {
namespace {

// SP[u] = [S[u] | P[u]]: 16-byte chunks, r a multiple of 8.
__global__ void __launch_bounds__(256) pack_cols_kernel(const __nv_bfloat16* __restrict__ S,
                                                        const __nv_bfloat16* __restrict__ P,
                                                        __nv_bfloat16* __restrict__ SP, int p,
                                                        int r) {
  const int per_row = 2 * r / 8;
  const long long e = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<long long>(p) * per_row) return;
  const int u = static_cast<int>(e / per_row);
  const int c = static_cast<int>(e - static_cast<long long>(u) * per_row) * 8;
  const __nv_bfloat16* src = c < r ? S + static_cast<size_t>(u) * r + c
                                   : P + static_cast<size_t>(u) * r + (c - r);
  *reinterpret_cast<uint4*>(SP + static_cast<size_t>(u) * 2 * r + c) =
      *reinterpret_cast<const uint4*>(src);
}

}  // namespace

cudaError_t launch_pack_cols(const void* S, const void* P, void* SP, int64_t p, int r,
                             cudaStream_t s) {
  if (r % 8 != 0) return cudaErrorInvalidValue;
  const long long chunks = p * (2 * r / 8);
  const int grid = static_cast<int>((chunks + 255) / 256);
  pack_cols_kernel<<<grid, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(S),
                                        static_cast<const __nv_bfloat16*>(P),
                                        static_cast<__nv_bfloat16*>(SP), static_cast<int>(p), r);
  return cudaGetLastError();
}

}  // namespace dprc
