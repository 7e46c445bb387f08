// Tensor-core (tcgen05 / TMEM / TMA) kernels of the Hutchinson and Hutch++
// norm estimators.
//
// Both estimators reduce to two contractions per sample i ("Efficient DP-SGD
// for LLMs with Randomized Clipping", papernotes.org, "Key design >
// Hutchinson": first the sketch G P, then Y = A^T (G P), then ||Y||_F^2):
//
//   row projection     W_i = X_i R        X_i [T][c] bf16, R [c][n]   -> T x n
//   column projection  Y_i = X_i^T W_i    X_i [T][c] bf16, W_i [T][n] -> c x n
//
// with (X, R) = (G, P) then (A, W) for Hutchinson.  Both stream X from HBM
// exactly once; their arithmetic intensity is ~n flop/byte, so they are
// HBM-bound and the tensor cores only have to keep up.
//
// Precision: X and R are bf16 (exact in fp32); accumulation is fp32 in TMEM.
// The fp32 sketch W is carried to the second contraction as two bf16 planes
// W = W_hi + W_lo (|W - W_hi - W_lo| <= 2^-17 |W|), multiplied as one MMA of
// width 2n whose two column halves are summed in the epilogue.

#include "common.cuh"
#include "internal.h"

namespace dprc {

namespace {

constexpr int kRowTile = 128;  // tokens per row-projection CTA (MMA M)
constexpr int kTileC = 64;     // c-columns per row-projection stage (128 B of bf16)
constexpr int kTileT = 64;     // T-rows per column-projection stage

__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Loads `NC` consecutive fp32 TMEM columns of this thread's lane.
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float* v) {
  static_assert(NC % 16 == 0, "columns in multiples of 16");
#pragma unroll
  for (int c0 = 0; c0 < NC; c0 += (NC % 32 == 0 ? 32 : 16)) {
    if constexpr (NC % 32 == 0) {
      float t[32];
      tmem_ld_32cols(taddr + c0, t);
#pragma unroll
      for (int j = 0; j < 32; ++j) v[c0 + j] = t[j];
    } else {
      float t[16];
      tmem_ld_16cols(taddr + c0, t);
#pragma unroll
      for (int j = 0; j < 16; ++j) v[c0 + j] = t[j];
    }
  }
}

// ===========================================================================
// Row projection: one CTA per 128-token tile, the whole c reduction in TMEM.
// Warp 0 lane 0: TMA producer.  Warp 1: TMEM allocator; its lane 0 issues
// the MMAs.  All four warps: epilogue (warp w owns TMEM lanes 32w..32w+31 =
// tokens t0+32w..t0+32w+31).
// ===========================================================================
template <int NMMA, bool HILO_IN>
struct RowCfg {
  static constexpr int kStages = 4;
  static constexpr int kXBytes = kRowTile * kTileC * 2;  // 16 KB
  static constexpr int kRBytes = kTileC * NMMA * 2;      // 2, 4 or 8 KB
  static constexpr int kStageBytes = kXBytes + kRBytes;
  static constexpr int kN = HILO_IN ? NMMA / 2 : NMMA;
  static constexpr int kTmemCols = NMMA < 32 ? 32 : NMMA;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 256;
  static_assert(NMMA == 16 || NMMA == 32 || NMMA == 64, "MN-major R atom is one swizzle row");
};

template <int NMMA, bool HILO_IN>
__global__ void __launch_bounds__(128, 1)
    tc_rowproj_kernel(const __grid_constant__ CUtensorMap map_x,
                      const __grid_constant__ CUtensorMap map_r, int T, int c, int r_batched,
                      int mtiles, __nv_bfloat16* __restrict__ W, long long tpad,
                      int* __restrict__ zero_ptr, int zero_ints) {
  using Cfg = RowCfg<NMMA, HILO_IN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_1024(smem_raw);
  uint8_t* sx = smem;
  uint8_t* sr = smem + Cfg::kStages * Cfg::kXBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sr + Cfg::kStages * Cfg::kRBytes);
  uint64_t* empty = full + Cfg::kStages;
  uint64_t* accf = empty + Cfg::kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accf + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int i = blockIdx.x / mtiles;
  const int t0 = (blockIdx.x % mtiles) * kRowTile;
  const int kc_n = (c + kTileC - 1) / kTileC;

  if (blockIdx.x == 0 && zero_ptr != nullptr)
    for (int z = threadIdx.x; z < zero_ints; z += blockDim.x) zero_ptr[z] = 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(accf, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_r);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0 && lane == 0) {
    int issued = 0;
    for (int kc = 0; kc < kc_n; ++kc) {
      const int s = kc % Cfg::kStages;
      const uint32_t ph = (kc / Cfg::kStages) & 1;
      if (!mbar_wait(&empty[s], ph ^ 1, DPRC_DEVERR_PIPE_EMPTY)) {
        *abort_flag = 1;
        break;
      }
      mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
      tma_load_3d(sx + s * Cfg::kXBytes, &map_x, &full[s], kc * kTileC, t0, i);
      tma_load_3d(sr + s * Cfg::kRBytes, &map_r, &full[s], 0, kc * kTileC, r_batched ? i : 0);
      ++issued;
    }
    // Let the copies this thread issued land before the CTA can exit.
    for (int kc = issued - 1; kc >= 0 && kc >= issued - Cfg::kStages; --kc)
      mbar_wait(&full[kc % Cfg::kStages], (kc / Cfg::kStages) & 1, DPRC_DEVERR_PIPE_FULL);
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = make_idesc_bf16(128, NMMA, false, true);
    constexpr uint32_t r_swz = swz_code_for_bytes(2 * NMMA);
    for (int kc = 0; kc < kc_n; ++kc) {
      const int s = kc % Cfg::kStages;
      const uint32_t ph = (kc / Cfg::kStages) & 1;
      if (!mbar_wait(&full[s], ph, DPRC_DEVERR_PIPE_FULL)) {
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
      const uint32_t xa = smem_u32(sx + s * Cfg::kXBytes);
      const uint32_t ra = smem_u32(sr + s * Cfg::kRBytes);
#pragma unroll
      for (int kk = 0; kk < kTileC / 16; ++kk) {
        // X tile: 128 token rows x 64 c, K-major, 128-byte swizzle.
        const uint64_t ad = make_sdesc(xa + kk * 32, 16, 1024, kSwz128);
        // R tile: 64 c rows x NMMA columns, MN-major, one swizzle atom wide;
        // 8-row atoms of 16*NMMA bytes, so a K=16 step is 32*NMMA bytes.
        const uint64_t bd = make_sdesc(ra + kk * 32 * NMMA, 16, 16 * NMMA, r_swz);
        umma_bf16(tmem, ad, bd, idesc, (kc | kk) != 0 ? 1u : 0u);
      }
      umma_commit(&empty[s]);
    }
    umma_commit(accf);
  }
  __syncwarp();

  // ---- epilogue: TMEM -> registers -> bf16 hi/lo planes of W ----
  const bool ok = __all_sync(0xffffffffu, mbar_wait(accf, 0, DPRC_DEVERR_ACCUM) && *abort_flag == 0);
  tc_fence_after();
  pdl_launch_dependents();
  if (ok) {
    float v[NMMA];
    tmem_ld_cols<NMMA>(tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
    const int t = t0 + warp * 32 + lane;
    if (t < T) {
      __nv_bfloat16* wi = W + static_cast<size_t>(i) * 2 * Cfg::kN * tpad + t;
#pragma unroll
      for (int j = 0; j < Cfg::kN; ++j) {
        const float y = HILO_IN ? v[j] + v[Cfg::kN + j] : v[j];
        __nv_bfloat16 hi, lo;
        split_hilo(y, hi, lo);
        wi[static_cast<size_t>(j) * tpad] = hi;
        wi[static_cast<size_t>(Cfg::kN + j) * tpad] = lo;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

// ===========================================================================
// Column projection, persistent stream-K over units (block b, T-tile kt),
// block b = (sample i, chunk of 256 output rows).  CTA j owns the contiguous
// unit range [j U / G, (j+1) U / G); each maximal run inside one block is a
// "segment" whose fp32 partial Y goes to a private slot.  A ticket per block
// finds the CTA that completes it; that CTA sums the block's partial slots in
// CTA order (deterministic), then applies the mode (norm / fp32 / hi-lo).
//
// Warp 0 lane 0: TMA producer.  Warp 1: TMEM allocator + MMA issuer.
// Warps 2..5: epilogue (warp w may access TMEM lanes 32*(w%4)...).  The
// accumulator is double-buffered in TMEM so MMAs of the next segment overlap
// the epilogue of the previous one.
// ===========================================================================
struct ColArgs {
  int T, c, nchunks, kt;
  long long units;
  int max_seg;
  float* part;
  int* tickets;
  int* sample_tickets;
  float* chunk_norms;
  int mode;
  float* n_out;
  int accumulate;
  int n_head;
  float w_tail;
  float* y_f32;
  __nv_bfloat16* y_hilo;
};

template <int NMMA>
struct ColCfg {
  static constexpr int kChunk = 256;
  static constexpr int kMB = kChunk / 128;
  static constexpr int kXBoxBytes = kTileT * 64 * 2;           // 64 T rows x 64 c = 8 KB
  static constexpr int kXBytes = kTileT * kChunk * 2;          // 32 KB
  static constexpr int kWBytes = NMMA * kTileT * 2;            // 4, 8 or 16 KB
  static constexpr int kStageBytes = kXBytes + kWBytes;
  static constexpr int kStages = NMMA >= 128 ? 4 : 5;
  static constexpr int kN = NMMA / 2;
  static constexpr int kAccCols = kMB * NMMA;
  static constexpr int kTmemCols = 2 * kAccCols;
  static constexpr int kSmem = kStages * kStageBytes + 1024 + 512;
  static_assert(kTmemCols <= 512, "TMEM has 512 columns");
};

__device__ __forceinline__ long long cta_of_unit(long long u, long long units, int G) {
  return ((u + 1) * G - 1) / units;
}

template <int NMMA>
__global__ void __launch_bounds__(192, 1)
    tc_colproj_kernel(const __grid_constant__ CUtensorMap map_x,
                      const __grid_constant__ CUtensorMap map_w, const ColArgs a) {
  using Cfg = ColCfg<NMMA>;
  constexpr int kN = Cfg::kN;
  extern __shared__ uint8_t smem_raw[];
  __shared__ int s_last;
  __shared__ float s_red[4];

  const int G = gridDim.x, j = blockIdx.x;
  const long long u0 = static_cast<long long>(j) * a.units / G;
  const long long u1 = static_cast<long long>(j + 1) * a.units / G;
  if (u0 >= u1) return;  // uniform across the CTA
  const int KT = a.kt;

  uint8_t* smem = align_1024(smem_raw);
  uint8_t* sx = smem;
  uint8_t* sw = smem + Cfg::kStages * Cfg::kXBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sw + Cfg::kStages * Cfg::kWBytes);
  uint64_t* empty = full + Cfg::kStages;
  uint64_t* accf = empty + Cfg::kStages;  // [2]
  uint64_t* acce = accf + 2;              // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_x);
    tma_prefetch_desc(&map_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // The sketch W and the cleared tickets come from the previous kernel.
  pdl_wait();

  if (warp == 0) {
    if (lane == 0) {
      long long issued = 0;
      for (long long u = u0; u < u1; ++u) {
        const int it = static_cast<int>(u - u0);
        const int s = it % Cfg::kStages;
        const uint32_t ph = (it / Cfg::kStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, DPRC_DEVERR_PIPE_EMPTY)) {
          *abort_flag = 1;
          break;
        }
        const long long b = u / KT;
        const int kt = static_cast<int>(u - b * KT);
        const int i = static_cast<int>(b / a.nchunks);
        const int ch = static_cast<int>(b - static_cast<long long>(i) * a.nchunks);
        mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
        uint8_t* xs = sx + s * Cfg::kXBytes;
#pragma unroll
        for (int q = 0; q < Cfg::kChunk / 64; ++q)
          tma_load_3d(xs + q * Cfg::kXBoxBytes, &map_x, &full[s], ch * Cfg::kChunk + q * 64,
                      kt * kTileT, i);
        tma_load_3d(sw + s * Cfg::kWBytes, &map_w, &full[s], kt * kTileT, 0, i);
        ++issued;
      }
      for (long long it = issued - 1; it >= 0 && it >= issued - Cfg::kStages; --it)
        mbar_wait(&full[it % Cfg::kStages], (it / Cfg::kStages) & 1, DPRC_DEVERR_PIPE_FULL);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc_bf16(128, NMMA, true, false);
      int seg = 0;
      for (long long u = u0; u < u1; ++u) {
        const int it = static_cast<int>(u - u0);
        const int s = it % Cfg::kStages;
        const uint32_t ph = (it / Cfg::kStages) & 1;
        const long long b = u / KT;
        const int kt = static_cast<int>(u - b * KT);
        const bool first = (u == u0) || (kt == 0);
        const bool last = (u == u1 - 1) || (kt == KT - 1);
        const int abuf = seg & 1;
        if (first) {
          if (!mbar_wait(&acce[abuf], ((seg >> 1) & 1) ^ 1, DPRC_DEVERR_ACCUM)) {
            *abort_flag = 1;
            break;
          }
          tc_fence_after();
        }
        if (!mbar_wait(&full[s], ph, DPRC_DEVERR_PIPE_FULL)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        const uint32_t xa = smem_u32(sx + s * Cfg::kXBytes);
        const uint32_t wa = smem_u32(sw + s * Cfg::kWBytes);
#pragma unroll
        for (int kk = 0; kk < kTileT / 16; ++kk) {
          // W tile: NMMA rows x 64 T, K-major, 128-byte swizzle.
          const uint64_t bd = make_sdesc(wa + kk * 32, 16, 1024, kSwz128);
#pragma unroll
          for (int mb = 0; mb < Cfg::kMB; ++mb) {
            // X tile: T rows of 64 c per 8 KB box; the operand X^T is MN-major
            // (c contiguous): atoms of 64 c x 8 T = 1 KB, SBO = 1 KB along T,
            // LBO = one box along c.  A K=16 step is two atoms (2 KB).
            const uint64_t ad = make_sdesc(xa + mb * 2 * Cfg::kXBoxBytes + kk * 2048,
                                           Cfg::kXBoxBytes, 1024, kSwz128);
            umma_bf16(tmem + abuf * Cfg::kAccCols + mb * NMMA, ad, bd, idesc,
                      (first && kk == 0) ? 0u : 1u);
          }
        }
        umma_commit(&empty[s]);
        if (last) {
          umma_commit(&accf[abuf]);
          ++seg;
        }
      }
    }
  } else {
    // ---------------- epilogue warps 2..5 ----------------
    const int ew = warp - 2;
    const int q = warp & 3;
    bool dead = false;
    const long long b_first = u0 / KT, b_last = (u1 - 1) / KT;
    int seg = 0;
    for (long long b = b_first; b <= b_last; ++b, ++seg) {
      const int abuf = seg & 1;
      if (!dead && !mbar_wait(&accf[abuf], (seg >> 1) & 1, DPRC_DEVERR_ACCUM)) dead = true;
      if (*abort_flag) dead = true;
      dead = __any_sync(0xffffffffu, dead);  // keep the warp's TMEM loads convergent
      tc_fence_after();
      float* slot = a.part + (static_cast<size_t>(j) * a.max_seg + seg) * Cfg::kChunk * kN;
      if (!dead) {
#pragma unroll 1
        for (int mb = 0; mb < Cfg::kMB; ++mb) {
          const int row = mb * 128 + q * 32 + lane;
          const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                              abuf * Cfg::kAccCols + mb * NMMA;
          float hi[kN], lo[kN];
          tmem_ld_cols<kN>(tb, hi);
          tmem_ld_cols<kN>(tb + kN, lo);
          float4* dst = reinterpret_cast<float4*>(slot + static_cast<size_t>(row) * kN);
#pragma unroll
          for (int c4 = 0; c4 < kN / 4; ++c4)
            dst[c4] = make_float4(hi[4 * c4] + lo[4 * c4], hi[4 * c4 + 1] + lo[4 * c4 + 1],
                                  hi[4 * c4 + 2] + lo[4 * c4 + 2], hi[4 * c4 + 3] + lo[4 * c4 + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[abuf]);
      __threadfence();
      named_bar_sync(1, 128);
      if (ew == 0 && lane == 0) {
        const long long lo_u = b * KT > u0 ? b * KT : u0;
        const long long hi_u = (b + 1) * KT < u1 ? (b + 1) * KT : u1;
        const int cnt = static_cast<int>(hi_u - lo_u);
        const int old = atomicAdd(&a.tickets[b], cnt);
        s_last = (!dead && old + cnt == KT) ? 1 : 0;
      }
      named_bar_sync(1, 128);
      if (s_last) {
        __threadfence();
        const int i = static_cast<int>(b / a.nchunks);
        const int ch = static_cast<int>(b - static_cast<long long>(i) * a.nchunks);
        const long long j_first = cta_of_unit(b * KT, a.units, G);
        const long long j_last = cta_of_unit((b + 1) * KT - 1, a.units, G);
        float sq = 0.f;
#pragma unroll 1
        for (int mb = 0; mb < Cfg::kMB; ++mb) {
          const int row = mb * 128 + ew * 32 + lane;
          const int grow = ch * Cfg::kChunk + row;
          float acc[kN];
#pragma unroll
          for (int t = 0; t < kN; ++t) acc[t] = 0.f;
          for (long long jj = j_first; jj <= j_last; ++jj) {
            const long long uj0 = jj * a.units / G;
            const int sj = static_cast<int>(b - uj0 / KT);
            const float4* src = reinterpret_cast<const float4*>(
                a.part + ((static_cast<size_t>(jj) * a.max_seg + sj) * Cfg::kChunk + row) * kN);
#pragma unroll
            for (int c4 = 0; c4 < kN / 4; ++c4) {
              const float4 v = __ldcg(src + c4);
              acc[4 * c4] += v.x;
              acc[4 * c4 + 1] += v.y;
              acc[4 * c4 + 2] += v.z;
              acc[4 * c4 + 3] += v.w;
            }
          }
          if (grow < a.c) {
            if (a.mode == kColprojNorm) {
#pragma unroll
              for (int t = 0; t < kN; ++t) sq += (t < a.n_head ? 1.f : a.w_tail) * acc[t] * acc[t];
            } else if (a.mode == kColprojF32) {
              float* dst = a.y_f32 + (static_cast<size_t>(i) * a.c + grow) * kN;
#pragma unroll
              for (int t = 0; t < kN; ++t) dst[t] = acc[t];
            } else {
              __nv_bfloat16* dst = a.y_hilo + (static_cast<size_t>(i) * a.c + grow) * 2 * kN;
#pragma unroll
              for (int t = 0; t < kN; ++t) split_hilo(acc[t], dst[t], dst[kN + t]);
            }
          }
        }
        if (a.mode == kColprojNorm) {
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
          if (lane == 0) s_red[ew] = sq;
          named_bar_sync(1, 128);
          if (ew == 0 && lane == 0) {
            const float tot = (s_red[0] + s_red[1]) + (s_red[2] + s_red[3]);
            a.chunk_norms[b] = tot;
            __threadfence();
            const int old = atomicAdd(&a.sample_tickets[i], 1);
            if (old == a.nchunks - 1) {
              __threadfence();
              float sum = 0.f;
              for (int c2 = 0; c2 < a.nchunks; ++c2)
                sum += __ldcg(&a.chunk_norms[static_cast<size_t>(i) * a.nchunks + c2]);
              a.n_out[i] = (a.accumulate ? a.n_out[i] : 0.f) + sum;
            }
          }
        }
      }
      named_bar_sync(1, 128);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
}

template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

template <int NMMA, bool HILO_IN>
cudaError_t rowproj_launch(const CUtensorMap& mx, const CUtensorMap& mr, int T, int c,
                           int r_batched, int B, void* W, long long tpad, int* zero_ptr,
                           int zero_ints, cudaStream_t s) {
  using Cfg = RowCfg<NMMA, HILO_IN>;
  auto kern = tc_rowproj_kernel<NMMA, HILO_IN>;
  cudaError_t e = set_smem(kern, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  const int mtiles = (T + kRowTile - 1) / kRowTile;
  kern<<<B * mtiles, 128, Cfg::kSmem, s>>>(mx, mr, T, c, r_batched, mtiles,
                                            static_cast<__nv_bfloat16*>(W), tpad, zero_ptr,
                                            zero_ints);
  return cudaGetLastError();
}

template <int NMMA>
cudaError_t colproj_launch(const CUtensorMap& mx, const CUtensorMap& mw, const ColArgs& args,
                           int grid, bool pdl, cudaStream_t s) {
  using Cfg = ColCfg<NMMA>;
  auto kern = tc_colproj_kernel<NMMA>;
  cudaError_t e = set_smem(kern, Cfg::kSmem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = Cfg::kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mx, mw, args);
}

}  // namespace

int colproj_stage_chunk() { return ColCfg<32>::kChunk; }

cudaError_t read_device_error(int32_t* out, bool reset) {
  int v = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_error, sizeof(int));
  if (e != cudaSuccess) return e;
  if (reset && v != 0) {
    const int z = 0;
    e = cudaMemcpyToSymbol(g_device_error, &z, sizeof(int));
  }
  *out = v;
  return e;
}

cudaError_t launch_tc_rowproj(const void* X, int64_t B, int64_t T, int64_t c, const void* R,
                              bool r_batched, int nmma, bool hilo_in, void* W, int64_t tpad,
                              int* zero_ptr, size_t zero_ints, cudaStream_t s) {
  CUtensorMap mx, mr;
  if (!make_tmap_3d_bf16(&mx, X, c, T, B, c, T * c, kTileC, kRowTile, 128))
    return cudaErrorInvalidValue;
  if (!make_tmap_3d_bf16(&mr, R, nmma, c, r_batched ? B : 1, nmma, c * nmma, nmma, kTileC,
                         2 * nmma))
    return cudaErrorInvalidValue;
  const int iT = static_cast<int>(T), ic = static_cast<int>(c), iB = static_cast<int>(B);
  const int zi = static_cast<int>(zero_ints);
  if (nmma == 16 && !hilo_in)
    return rowproj_launch<16, false>(mx, mr, iT, ic, r_batched, iB, W, tpad, zero_ptr, zi, s);
  if (nmma == 32 && !hilo_in)
    return rowproj_launch<32, false>(mx, mr, iT, ic, r_batched, iB, W, tpad, zero_ptr, zi, s);
  if (nmma == 64 && !hilo_in)
    return rowproj_launch<64, false>(mx, mr, iT, ic, r_batched, iB, W, tpad, zero_ptr, zi, s);
  if (nmma == 32 && hilo_in)
    return rowproj_launch<32, true>(mx, mr, iT, ic, r_batched, iB, W, tpad, zero_ptr, zi, s);
  if (nmma == 64 && hilo_in)
    return rowproj_launch<64, true>(mx, mr, iT, ic, r_batched, iB, W, tpad, zero_ptr, zi, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_tc_colproj(const void* X, int64_t B, int64_t T, int64_t c, const void* W,
                              int64_t tpad, int n, const ColprojPlan& plan, char* ws,
                              ColprojMode mode, float* n_out, int accumulate, int n_head,
                              float w_tail, float* y_f32, void* y_hilo, bool pdl,
                              cudaStream_t s) {
  const int nmma = 2 * n;
  CUtensorMap mx, mw;
  if (!make_tmap_3d_bf16(&mx, X, c, T, B, c, T * c, 64, kTileT, 128))
    return cudaErrorInvalidValue;
  if (!make_tmap_3d_bf16(&mw, W, T, nmma, B, tpad, nmma * tpad, kTileT, nmma, 128))
    return cudaErrorInvalidValue;
  ColArgs a;
  a.T = static_cast<int>(T);
  a.c = static_cast<int>(c);
  a.nchunks = plan.nchunks;
  a.kt = plan.kt;
  a.units = plan.units;
  a.max_seg = plan.max_seg;
  a.part = reinterpret_cast<float*>(ws + plan.part_off);
  a.tickets = reinterpret_cast<int*>(ws + plan.tick_off);
  a.sample_tickets = reinterpret_cast<int*>(ws + plan.stick_off);
  a.chunk_norms = reinterpret_cast<float*>(ws + plan.cnorm_off);
  a.mode = mode;
  a.n_out = n_out;
  a.accumulate = accumulate;
  a.n_head = n_head;
  a.w_tail = w_tail;
  a.y_f32 = y_f32;
  a.y_hilo = static_cast<__nv_bfloat16*>(y_hilo);
  if (nmma == 32) return colproj_launch<32>(mx, mw, a, plan.grid, pdl, s);
  if (nmma == 64) return colproj_launch<64>(mx, mw, a, plan.grid, pdl, s);
  if (nmma == 128) return colproj_launch<128>(mx, mw, a, plan.grid, pdl, s);
  return cudaErrorInvalidValue;
}

}  // namespace dprc
