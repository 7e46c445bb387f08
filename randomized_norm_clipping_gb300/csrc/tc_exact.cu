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
  uint64_t* drain = acce + 2;           // MMA thread: all its MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 3);
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
    mbar_init(drain, 1);
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
      bool ok = true, issued = false;
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
          issued = true;
        }
        if (ok) umma_commit(&accf[abuf]);
      }
      // on every path out of the loop: no MMA still writes the tensor memory
      // the CTA releases
      if (issued) umma_drain(drain, kWaitLimitNs);
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
      if (ew == 0 && lane == 0 && ok && DPRC_IN(blockIdx.x + j * gridDim.x < a.ntiles))
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

// ---------------------------------------------------------------------------
// Ghost form on tensor cores.
//
//   n_i = sum_{t,s} (A_i A_i^T)_{ts} (G_i G_i^T)_{ts}
//       = sum over 128-token blocks tb <= sb of w(tb, sb) <S_A[tb, sb], S_G[tb, sb]>
//
// with S_A = A_i A_i^T, S_G = G_i G_i^T and w = 1 on the diagonal, 2 off it
// (both Grams are symmetric).  A unit of work is one row block tb of one
// sample against a span of up to W column blocks starting at sb0 = tb + W m:
// the Gram tiles S_A[tb, span] (K = d) and S_G[tb, span] (K = p), 128 x 128 W
// each, accumulated in fp32 TMEM one after the other by tcgen05.mma from
// K-major operands (A [T][d] and G [T][p] as stored: the feature axis is the
// contraction axis).  Eight epilogue warps copy S_A into registers as soon as
// it is complete, which frees its columns for the next unit, and take the
// weighted dot product with S_G when that completes; the epilogue of one unit
// thus overlaps the MMAs of the next without a second accumulator.  One
// partial per unit; the finishing kernel sums a sample's partials in index
// order (deterministic).  Ragged T reads zero rows past the end (TMA fill),
// ragged d and p zero columns, which add nothing.
//
// The units of one sample are numbered by r = nt - tb ascending (nt blocks
// per sample): row block tb has ceil(r / W) spans, so r <= R holds
// S_W(R) = sum_{r <= R} ceil(r / W) units, R (R + 1) / 2 for W = 1 and
// floor((R + 1)^2 / 4) for W = 2.
// ---------------------------------------------------------------------------
constexpr int kGhRows = 128;                 // tokens per block (MMA M)
constexpr int kGhK = 64;                     // features per stage (one 128 B swizzle row)
constexpr int kGhBox = kGhRows * kGhK * 2;   // one 128-token x 64-feature box, 16 KB
constexpr int kGhRing = 192 * 1024;
constexpr int kGhEpiWarps = 8;
constexpr int kGhThreads = 64 + 32 * kGhEpiWarps;

template <int W>
struct GhCfg {
  static constexpr int kStage = (1 + W) * kGhBox;   // row block + span
  static constexpr int kStages = kGhRing / kStage;  // 4 (W = 2) or 6 (W = 1)
  static constexpr int kN = kGhRows * W;            // Gram tile width (MMA N)
  static constexpr int kTmemCols = 2 * kN;          // S_A | S_G
  static constexpr int kHalf = kN / 2;              // columns per epilogue warp
  static constexpr int kSmem = kStages * kStage + 1024 + 256;
};

__host__ __device__ inline long long ghost_span_units(long long R, int W) {
  return W == 1 ? R * (R + 1) / 2 : (R + 1) * (R + 1) / 4;
}

struct GhostArgs {
  int nt;                     // 128-token blocks per sample
  int nd, np;                 // 64-feature stages of A and of G per unit
  long long per_sample;       // units per sample, S_W(nt)
  long long nunits;           // B * per_sample
  float* partials;            // [nunits]
  unsigned long long* next;   // work counter (zero on entry, zero on exit)
  unsigned int* done;         // CTAs finished (zero on entry, zero on exit)
};

struct GhostUnit {
  int i, tb, sb0, width, m;
};

// Unit g of the queue: sample g / per_sample; within the sample the units run
// from r = nt down to r = 1 (the last units of a sample are its smallest).
template <int W>
__device__ __forceinline__ GhostUnit ghost_unit(const GhostArgs& a, long long g) {
  GhostUnit u;
  u.i = static_cast<int>(g / a.per_sample);
  const long long ul = a.per_sample - 1 - (g - static_cast<long long>(u.i) * a.per_sample);
  // smallest R with S_W(R) > ul: a float estimate, then exact integer steps
  const float x = W == 1 ? (sqrtf(8.f * static_cast<float>(ul) + 1.f) - 1.f) * 0.5f
                         : 2.f * sqrtf(static_cast<float>(ul)) - 1.f;
  long long R = x > 1.f ? static_cast<long long>(x) : 1;
  while (ghost_span_units(R, W) <= ul) ++R;
  while (R > 1 && ghost_span_units(R - 1, W) > ul) --R;
  u.m = static_cast<int>(ul - ghost_span_units(R - 1, W));
  u.tb = a.nt - static_cast<int>(R);
  u.sb0 = u.tb + W * u.m;
  u.width = a.nt - u.sb0 < W ? a.nt - u.sb0 : W;
  return u;
}

// Persistent CTAs take units from a global counter in queue order (sample by
// sample, so the CTAs at work share a few samples' A and G in L2), which
// evens out the unequal units (spans clipped at the last block) better than a
// fixed assignment.  Which CTA computes a unit does not change its partial,
// so the result stays bitwise repeatable.  The producer announces each unit
// in a tag beside the stage it loads; the MMA thread passes it on to the
// epilogue through a two-slot mailbox; -1 ends both.
template <int W>
__global__ void __launch_bounds__(kGhThreads, 1)
    tc_ghost_norm_kernel(const __grid_constant__ CUtensorMap map_a,
                         const __grid_constant__ CUtensorMap map_g, const GhostArgs a) {
  using Cfg = GhCfg<W>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_red[kGhEpiWarps];
  __shared__ long long stage_unit[Cfg::kStages];
  __shared__ long long epi_unit[2];
  __shared__ volatile int epi_stop;

  uint8_t* ring = align_1024(smem_raw);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + Cfg::kStages * Cfg::kStage);
  uint64_t* empty = full + Cfg::kStages;
  uint64_t* a_full = empty + Cfg::kStages;  // S_A complete
  uint64_t* a_free = a_full + 1;            // S_A copied out of TMEM
  uint64_t* g_full = a_free + 1;            // S_G complete
  uint64_t* g_free = g_full + 1;            // S_G consumed
  uint64_t* mail = g_free + 1;              // [2] epilogue mailbox filled
  uint64_t* drain = mail + 2;               // MMA thread: all its MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mail + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = a.nd + a.np;  // stages per unit

  if (threadIdx.x == 0) {
    for (int s = 0; s < Cfg::kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(a_full, 1);
    mbar_init(g_full, 1);
    mbar_init(a_free, kGhEpiWarps);
    mbar_init(g_free, kGhEpiWarps);
    mbar_init(&mail[0], 1);
    mbar_init(&mail[1], 1);
    mbar_init(drain, 1);
    fence_mbar_init();
    *abort_flag = 0;
    epi_stop = 0;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_g);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      long long it = 0;
      // the next unit is claimed two stages before the current one is fully
      // issued: the atomic's round trip overlaps those loads, and a unit is
      // not held long enough to unbalance the end of the queue
      long long g_next = static_cast<long long>(atomicAdd(a.next, 1ull));
      while (true) {
        const long long g = g_next;
        const bool last = g >= a.nunits;
        const GhostUnit u = ghost_unit<W>(a, last ? 0 : g);
        const int claim_at = nk > 2 ? nk - 2 : 0;
        bool ok = true;
        for (int f = 0; f < (last ? 1 : nk); ++f, ++it) {
          if (!last && f == claim_at) g_next = static_cast<long long>(atomicAdd(a.next, 1ull));
          const int s = static_cast<int>(it % Cfg::kStages);
          const uint32_t ph = static_cast<uint32_t>(it / Cfg::kStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, DPRC_DEVERR_PIPE_EMPTY)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          stage_unit[s] = last ? -1 : g;  // published by the arrive below
          if (last) {
            mbar_arrive(&full[s]);
            break;
          }
          const bool is_a = f < a.nd;
          const CUtensorMap* map = is_a ? &map_a : &map_g;
          const int x = (is_a ? f : f - a.nd) * kGhK;
          uint8_t* st = ring + s * Cfg::kStage;
          mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>((1 + u.width) * kGhBox));
          tma_load_3d(st, map, &full[s], x, u.tb * kGhRows, u.i);
          for (int h = 0; h < u.width; ++h)
            tma_load_3d(st + (1 + h) * kGhBox, map, &full[s], x, (u.sb0 + h) * kGhRows, u.i);
        }
        if (last || !ok) {
          if (last && ok) ++it;
          break;
        }
      }
      // let the copies this thread issued land before the CTA can exit
      for (long long k = it - 1; k >= 0 && k >= it - Cfg::kStages; --k)
        mbar_wait(&full[k % Cfg::kStages], (k / Cfg::kStages) & 1, DPRC_DEVERR_PIPE_FULL);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_w = make_idesc_bf16(kGhRows, Cfg::kN, false, false);
      constexpr uint32_t idesc_1 = make_idesc_bf16(kGhRows, kGhRows, false, false);
      long long it = 0;
      bool issued = false;
      for (long long j = 0;; ++j) {
        // the unit's first stage names it
        const int s0 = static_cast<int>(it % Cfg::kStages);
        const uint32_t ph0 = static_cast<uint32_t>(it / Cfg::kStages) & 1;
        bool ok = mbar_wait(&full[s0], ph0, DPRC_DEVERR_PIPE_FULL);
        const long long g = ok ? stage_unit[s0] : -1;
        const uint32_t par = static_cast<uint32_t>(j & 1);
        // the epilogue has copied out S_A of unit j - 1, so it is done with
        // mailbox slot j & 1 and with S_A's columns
        ok = ok && mbar_wait(a_free, par ^ 1, DPRC_DEVERR_ACCUM);
        epi_unit[j & 1] = ok ? g : -1;
        mbar_arrive(&mail[j & 1]);
        if (!ok || g < 0) {
          if (!ok) *abort_flag = 1;
          break;
        }
        const GhostUnit u = ghost_unit<W>(a, g);
        const uint32_t idesc = u.width == W ? idesc_w : idesc_1;
        for (int part = 0; part < 2 && ok; ++part) {
          if (part == 1 && !mbar_wait(g_free, par ^ 1, DPRC_DEVERR_ACCUM)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const int f0 = part == 0 ? 0 : a.nd, f1 = part == 0 ? a.nd : nk;
          const uint32_t dst = tmem + static_cast<uint32_t>(part * Cfg::kN);
          for (int f = f0; f < f1; ++f, ++it) {
            const int s = static_cast<int>(it % Cfg::kStages);
            const uint32_t ph = static_cast<uint32_t>(it / Cfg::kStages) & 1;
            if (!mbar_wait(&full[s], ph, DPRC_DEVERR_PIPE_FULL)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t ta = smem_u32(ring + s * Cfg::kStage);
#pragma unroll
            for (int kk = 0; kk < kGhK / 16; ++kk) {
              // both operands K-major, 128-byte swizzle: 8-row atoms 1 KB
              // apart (SBO), a K = 16 step is 32 B along the swizzled row
              const uint64_t ad = make_sdesc(ta + kk * 32, 16, 1024, kSwz128);
              const uint64_t bd = make_sdesc(ta + kGhBox + kk * 32, 16, 1024, kSwz128);
              umma_bf16(dst, ad, bd, idesc, (f == f0 && kk == 0) ? 0u : 1u);
            }
            umma_commit(&empty[s]);
            issued = true;
          }
          if (ok) umma_commit(part == 0 ? a_full : g_full);
        }
        if (!ok) {
          *abort_flag = 1;
          break;
        }
      }
      // on every path out of the loop: no MMA still writes the tensor memory
      // the CTA releases
      if (issued) umma_drain(drain, kWaitLimitNs);
    }
  } else {
    // ---------------- epilogue warps 2 .. 9 ----------------
    // Every epilogue warp runs the same iterations: whether to stop is read
    // from one shared flag between the two named barriers of an iteration.
    constexpr int kChunks = Cfg::kHalf / 32;
    const int ew = warp - 2;
    const int q = warp & 3;    // TMEM lane quadrant this warp may read
    const int half = ew >> 2;  // which half of the tile's columns
    for (long long j = 0;; ++j) {
      const uint32_t par = static_cast<uint32_t>(j & 1);
      const bool got = mbar_wait(&mail[j & 1], static_cast<uint32_t>((j >> 1) & 1),
                                 DPRC_DEVERR_ACCUM);
      const long long g = got ? epi_unit[j & 1] : -1;
      const bool have = __all_sync(0xffffffffu, g >= 0);  // a unit, not the end mark
      float w = 0.f;
      uint32_t tb = 0;
      bool live = have;
      if (have) {
        const GhostUnit u = ghost_unit<W>(a, g);
        // weight of this warp's columns: the diagonal block counts once,
        // blocks above it twice, columns past the span not at all
        if (W == 2)
          w = half == 0 ? (u.m == 0 ? 1.f : 2.f) : (u.width == 2 ? 2.f : 0.f);
        else
          w = u.m == 0 ? 1.f : 2.f;
        tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(half * Cfg::kHalf);
        live = mbar_wait(a_full, par, DPRC_DEVERR_ACCUM) && *abort_flag == 0;
      }
      live = __all_sync(0xffffffffu, live);  // keep the warp's TMEM loads convergent
      tc_fence_after();
      float ra[kChunks][32];
      if (live && w != 0.f) {
#pragma unroll
        for (int c = 0; c < kChunks; ++c) tmem_ld_32cols(tb + c * 32, ra[c]);
      }
      tc_fence_before();
      __syncwarp();
      if (have && lane == 0) mbar_arrive(a_free);
      live = live && mbar_wait(g_full, par, DPRC_DEVERR_ACCUM) && *abort_flag == 0;
      live = __all_sync(0xffffffffu, live);
      tc_fence_after();
      float s0 = 0.f, s1 = 0.f;
      if (live && w != 0.f) {
#pragma unroll
        for (int c = 0; c < 2 * kChunks; ++c) {
          float v[16];  // 16 columns at a time keeps S_A's registers from spilling
          tmem_ld_16cols(tb + Cfg::kN + c * 16, v);
#pragma unroll
          for (int t = 0; t < 16; t += 2) {
            s0 = fmaf(ra[c >> 1][(c & 1) * 16 + t], v[t], s0);
            s1 = fmaf(ra[c >> 1][(c & 1) * 16 + t + 1], v[t + 1], s1);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (have && lane == 0) mbar_arrive(g_free);
      float sq = s0 + s1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      if (lane == 0) {
        s_red[ew] = sq * w;
        if (!live) epi_stop = 1;  // the end mark, or a wait that ran out
      }
      named_bar_sync(1, 32 * kGhEpiWarps);
      const bool stop = epi_stop != 0;
      if (ew == 0 && lane == 0 && !stop && DPRC_IN(g >= 0 && g < a.nunits)) {
        float tot = 0.f;
#pragma unroll
        for (int e = 0; e < kGhEpiWarps; ++e) tot += s_red[e];
        a.partials[g] = tot;
      }
      named_bar_sync(1, 32 * kGhEpiWarps);
      if (stop) break;
    }
  }

  __syncwarp();  // reconverge each warp before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
  // the last CTA out leaves the counters zero for the next call
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.done, 1u) == gridDim.x - 1) {
      atomicExch(a.next, 0ull);
      atomicExch(a.done, 0u);
    }
  }
}

template <int W>
cudaError_t set_ghost_smem_once() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> done[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(tc_ghost_norm_kernel<W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           GhCfg<W>::kSmem);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDev) done[dev].store(1, std::memory_order_release);
  return e;
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

int64_t ghost_partials(int64_t B, int64_t T, int W) {
  return B * ghost_span_units((T + kGhRows - 1) / kGhRows, W);
}

cudaError_t launch_tc_exact_ghost(const void* A, const void* G, int64_t B, int64_t T, int64_t d,
                                  int64_t p, int W, void* counters, float* partials,
                                  float* n_out, int accumulate, cudaStream_t s) {
  if (W != 1 && W != 2) return cudaErrorInvalidValue;
  CUtensorMap ma, mg;
  if (!make_tmap_3d_bf16(&ma, A, d, T, B, d, T * d, kGhK, kGhRows, 128))
    return cudaErrorInvalidValue;
  if (!make_tmap_3d_bf16(&mg, G, p, T, B, p, T * p, kGhK, kGhRows, 128))
    return cudaErrorInvalidValue;
  GhostArgs a;
  a.nt = static_cast<int>((T + kGhRows - 1) / kGhRows);
  a.nd = static_cast<int>((d + kGhK - 1) / kGhK);
  a.np = static_cast<int>((p + kGhK - 1) / kGhK);
  a.per_sample = ghost_span_units(a.nt, W);
  a.nunits = B * a.per_sample;
  a.partials = partials;
  a.next = static_cast<unsigned long long*>(counters);
  a.done = reinterpret_cast<unsigned int*>(a.next + 1);
  const long long grid = a.nunits < device_sm_count() ? a.nunits : device_sm_count();
  cudaError_t e = W == 1 ? set_ghost_smem_once<1>() : set_ghost_smem_once<2>();
  if (e != cudaSuccess) return e;
  if (W == 1)
    tc_ghost_norm_kernel<1><<<static_cast<unsigned>(grid), kGhThreads, GhCfg<1>::kSmem, s>>>(
        ma, mg, a);
  else
    tc_ghost_norm_kernel<2><<<static_cast<unsigned>(grid), kGhThreads, GhCfg<2>::kSmem, s>>>(
        ma, mg, a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_partials_finish(partials, B, a.per_sample, n_out, accumulate, s);
}

}  // namespace dprc
