// Exact per-sample gradient norm on tensor cores, direct form.
//
// The per-sample weight gradient of a linear layer is A_i^T G_i (d x p), and
// its squared Frobenius norm is the quantity the clipping needs
// ("Efficient DP-SGD for LLMs with Randomized Clipping", papernotes.org,
// "Key design > Hutchinson": n_i = ||A_i^T G_i||_F^2 = trace(G_i^T A_i A_i^T G_i)).
// The pages compare two exact ways of getting it: forming A_i^T G_i (O(T d p)
// flops per sample, what they call full gradient computation) and the ghost
// form sum_{t,s} (A A^T)_{ts} (G G^T)_{ts} (O(T^2 (d + p))) ("Related work";
// gist.science summary, "Complexiteitsreductie").  This kernel is the first:
//
//   n_i = sum over tiles (m, n) of || (A_i^T G_i)[128 m .., 256 n ..] ||^2
//
// with each 128 x 256 tile of A_i^T G_i accumulated over T in fp32 TMEM by
// tcgen05.mma (bf16 operands, both MN-major: A [T][d] and G [T][p] are read
// as stored, d and p contiguous) and squared and summed by the epilogue, so
// the d x p matrix is never stored.  Each tile writes one partial; a
// finishing kernel sums a sample's partials in index order (deterministic).
//
// Persistent grid (one CTA per SM), tiles taken in sample-major order with a
// stride of the grid size, so the CTAs running at one time share one or two
// samples' A and G in L2.  Warp 0: TMA producer; warp 1: TMEM allocator and
// MMA issuer; warps 2..5: epilogue.  The 256-column accumulator is double
// buffered (all 512 TMEM columns), so a tile's epilogue overlaps the next
// tile's MMAs.

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace dprc {

namespace {

constexpr int kFgcM = 128;     // rows of d per tile (MMA M)
constexpr int kFgcN = 256;     // columns of p per tile (MMA N)
constexpr int kFgcK = 64;      // tokens per pipeline stage
constexpr int kFgcStages = 4;
constexpr int kABoxBytes = kFgcK * 64 * 2;            // 64 tokens x 64 d, 8 KB
constexpr int kABytes = (kFgcM / 64) * kABoxBytes;    // 16 KB
constexpr int kBBoxBytes = kFgcK * 64 * 2;            // 64 tokens x 64 p, 8 KB
constexpr int kBBytes = (kFgcN / 64) * kBBoxBytes;    // 32 KB
constexpr int kFgcStageBytes = kABytes + kBBytes;     // 48 KB
constexpr int kFgcTmemCols = 2 * kFgcN;               // 512
constexpr int kFgcSmem = kFgcStages * kFgcStageBytes + 1024 + 256;

struct FgcArgs {
  int T, mt, nt;        // tokens; d-tiles and p-tiles per sample
  long long ntiles;     // B * mt * nt
  float* partials;      // [ntiles]
};

__global__ void __launch_bounds__(192, 1)
    tc_fgc_norm_kernel(const __grid_constant__ CUtensorMap map_a,
                       const __grid_constant__ CUtensorMap map_g, const FgcArgs a) {
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_red[4];

  uint8_t* smem = align_1024(smem_raw);
  uint8_t* sa = smem;
  uint8_t* sb = smem + kFgcStages * kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sb + kFgcStages * kBBytes);
  uint64_t* empty = full + kFgcStages;
  uint64_t* accf = empty + kFgcStages;  // [2]
  uint64_t* acce = accf + 2;            // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nu = (a.T + kFgcK - 1) / kFgcK;  // K units per tile
  // tiles of this CTA: blockIdx.x, blockIdx.x + gridDim.x, ...
  const long long my_tiles =
      a.ntiles > blockIdx.x ? (a.ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kFgcStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);
    }
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_g);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kFgcTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0 && my_tiles > 0) {
      long long it = 0;
      bool ok = true;
      for (long long j = 0; j < my_tiles && ok; ++j) {
        const long long tile = blockIdx.x + j * gridDim.x;
        const int i = static_cast<int>(tile / (static_cast<long long>(a.mt) * a.nt));
        const int rem = static_cast<int>(tile - static_cast<long long>(i) * a.mt * a.nt);
        const int m = rem / a.nt, n = rem - (rem / a.nt) * a.nt;
        for (int u = 0; u < nu; ++u, ++it) {
          const int s = static_cast<int>(it % kFgcStages);
          const uint32_t ph = static_cast<uint32_t>(it / kFgcStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, DPRC_DEVERR_PIPE_EMPTY)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], kFgcStageBytes);
#pragma unroll
          for (int h = 0; h < kFgcM / 64; ++h)
            tma_load_3d(sa + s * kABytes + h * kABoxBytes, &map_a, &full[s],
                        m * kFgcM + h * 64, u * kFgcK, i);
#pragma unroll
          for (int h = 0; h < kFgcN / 64; ++h)
            tma_load_3d(sb + s * kBBytes + h * kBBoxBytes, &map_g, &full[s],
                        n * kFgcN + h * 64, u * kFgcK, i);
        }
      }
      // let the copies this thread issued land before the CTA can exit
      for (long long k = it - 1; k >= 0 && k >= it - kFgcStages; --k)
        mbar_wait(&full[k % kFgcStages], (k / kFgcStages) & 1, DPRC_DEVERR_PIPE_FULL);
    }
  } else if (warp == 1) {
    if (lane == 0 && my_tiles > 0) {
      constexpr uint32_t idesc = make_idesc_bf16(kFgcM, kFgcN, true, true);
      long long it = 0;
      bool ok = true;
      for (long long j = 0; j < my_tiles && ok; ++j) {
        const int abuf = static_cast<int>(j & 1);
        if (!mbar_wait(&acce[abuf], static_cast<uint32_t>((j >> 1) & 1) ^ 1, DPRC_DEVERR_ACCUM)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        for (int u = 0; u < nu; ++u, ++it) {
          const int s = static_cast<int>(it % kFgcStages);
          const uint32_t ph = static_cast<uint32_t>(it / kFgcStages) & 1;
          if (!mbar_wait(&full[s], ph, DPRC_DEVERR_PIPE_FULL)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t aa = smem_u32(sa + s * kABytes);
          const uint32_t ba = smem_u32(sb + s * kBBytes);
#pragma unroll
          for (int kk = 0; kk < kFgcK / 16; ++kk) {
            // Both operands MN-major with a 128-byte swizzle: a K = 16 step is
            // 16 token rows of 128 B; 8-row atoms 1 KB apart (SBO); 64-wide
            // atoms along M or N one TMA box apart (LBO).
            const uint64_t ad = make_sdesc(aa + kk * 2048, kABoxBytes, 1024, kSwz128);
            const uint64_t bd = make_sdesc(ba + kk * 2048, kBBoxBytes, 1024, kSwz128);
            umma_bf16(tmem + abuf * kFgcN, ad, bd, idesc, (u == 0 && kk == 0) ? 0u : 1u);
          }
          umma_commit(&empty[s]);
        }
        if (ok) umma_commit(&accf[abuf]);
      }
    }
  } else {
    // ---------------- epilogue warps 2..5 ----------------
    const int ew = warp - 2;
    const int q = warp & 3;  // TMEM lane quadrant this warp may read
    bool ok = true;
    for (long long j = 0; j < my_tiles; ++j) {
      const int abuf = static_cast<int>(j & 1);
      bool live = ok && mbar_wait(&accf[abuf], static_cast<uint32_t>((j >> 1) & 1),
                                  DPRC_DEVERR_ACCUM) &&
                  *abort_flag == 0;
      live = __all_sync(0xffffffffu, live);  // keep the warp's TMEM loads convergent
      if (!live) ok = false;
      tc_fence_after();
      float sq = 0.f;
      if (live) {
        const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + abuf * kFgcN;
#pragma unroll 1
        for (int c0 = 0; c0 < kFgcN; c0 += 32) {
          float v[32];
          tmem_ld_32cols(tb + c0, v);
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int t = 0; t < 32; t += 2) {
            s0 = fmaf(v[t], v[t], s0);
            s1 = fmaf(v[t + 1], v[t + 1], s1);
          }
          sq += s0 + s1;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[abuf]);
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      if (lane == 0) s_red[ew] = sq;
      named_bar_sync(1, 128);
      if (ew == 0 && lane == 0 && ok)
        a.partials[blockIdx.x + j * gridDim.x] = (s_red[0] + s_red[1]) + (s_red[2] + s_red[3]);
      named_bar_sync(1, 128);
    }
  }

  __syncwarp();  // reconverge each warp before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kFgcTmemCols);
  }
}

cudaError_t set_fgc_smem_once() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> done[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(tc_fgc_norm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kFgcSmem);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDev) done[dev].store(1, std::memory_order_release);
  return e;
}

}  // namespace

cudaError_t read_device_error_exact(int32_t* out, bool reset) {
  return read_tu_device_error(out, reset);
}

int64_t fgc_partials(int64_t B, int64_t d, int64_t p) {
  return B * ((d + kFgcM - 1) / kFgcM) * ((p + kFgcN - 1) / kFgcN);
}

cudaError_t launch_tc_exact_direct(const void* A, const void* G, int64_t B, int64_t T, int64_t d,
                                   int64_t p, float* partials, float* n_out, int accumulate,
                                   cudaStream_t s) {
  CUtensorMap ma, mg;
  if (!make_tmap_3d_bf16(&ma, A, d, T, B, d, T * d, 64, kFgcK, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_3d_bf16(&mg, G, p, T, B, p, T * p, 64, kFgcK, 128)) return cudaErrorInvalidValue;
  FgcArgs a;
  a.T = static_cast<int>(T);
  a.mt = static_cast<int>((d + kFgcM - 1) / kFgcM);
  a.nt = static_cast<int>((p + kFgcN - 1) / kFgcN);
  a.ntiles = fgc_partials(B, d, p);
  a.partials = partials;
  cudaError_t e = set_fgc_smem_once();
  if (e != cudaSuccess) return e;
  const long long grid = a.ntiles < device_sm_count() ? a.ntiles : device_sm_count();
  tc_fgc_norm_kernel<<<static_cast<unsigned>(grid), 192, kFgcSmem, s>>>(ma, mg, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_partials_finish(partials, B, static_cast<int64_t>(a.mt) * a.nt, n_out, accumulate,
                                s);
}

}  // namespace dprc
