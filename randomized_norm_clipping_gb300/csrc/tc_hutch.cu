// One-launch Hutchinson estimate on tensor cores:
//
//   n_i (+)= || A_i^T (G_i P) ||_F^2
//
// ("Efficient DP-SGD for LLMs with Randomized Clipping", papernotes.org,
// "Key design > Hutchinson": the sketch G P first, then Y = A^T (G P), then
// its squared Frobenius norm).
//
// The two contractions of tc_proj.cu (the sketch W_i = G_i P and the
// projection Y_i = A_i^T W_i) run as two phases of one persistent kernel
// instead of two launches:
//
//   phase 1  every CTA takes sketch blocks (128 tokens of one sample) and
//            writes W_i as bf16 hi/lo planes [B][2k][T_pad]; after each block
//            it adds one to the per-sample counter ready[i] (release);
//   phase 2  every CTA takes projection blocks (sample i, 128 rows of d);
//            its TMA producer issues the A tiles at once, waits until
//            ready[i] has reached the number of sketch blocks of sample i
//            (acquire), then loads the W tiles; the epilogue squares Y and
//            a per-sample ticket sums the blocks in order into n_i.
//
// This removes the second launch, the wait for the first grid to drain and
// the projection's pipeline ramp, and lets the A stream of phase 2 start
// while the last sketch tiles are still in flight.  The cross-CTA waits are
// safe because the launch is cooperative (every CTA is resident) and phase 1
// never waits on another CTA; every wait is bounded (2 s) and records a code
// in the device error word when it runs out.
//
// Each phase assigns blocks either whole, strided over the CTAs, or one at a
// time to a thread-block cluster whose CTAs split the block's units and
// reduce the fp32 partials through distributed shared memory (credits make
// the receive buffer reusable across blocks and phases).
//
// Counters: the last block of sample i (ticket) resets ready[i] and the
// ticket to zero, so the counter block is zero after every call and must be
// zero before the first.
//
// One CTA per SM (the driver counts tensor-memory kernels at one CTA per SM,
// and a cooperative launch cannot exceed that), with a 192 KB shared-memory
// ring so that each SM keeps as many bytes in flight as two CTAs of the
// two-kernel path.  Both phases use four slots of R/4 bytes; phase-2 slot c
// overlays phase-1 slot c and is first filled once that has been consumed.
// A sketch stage is 128 tokens x 128 p of G (two TMA boxes, 256 contiguous
// bytes per row) plus 128 rows of P; a projection stage 128 tokens x 128 d
// of A plus the matching 128 tokens of the sketch.  TMEM: phase-1 accumulators (2 x 32
// columns) and phase-2 accumulators (2 x 2k columns), 256 columns.

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace dprc {

namespace {

constexpr int kTok = 128;   // tokens per sketch block; tokens per projection unit
constexpr int kCol = 128;   // columns of p per sketch unit (two 64-column boxes)
constexpr int kRows = 128;  // rows of d per projection block

template <int K>
struct HCfg {
  static constexpr int kNR = K;       // sketch MMA N
  static constexpr int kNC = 2 * K;   // projection MMA N (hi | lo)
  static constexpr int kRowStages = 4;
  static constexpr int kColStages = 4;
  static constexpr int kRowGBox = kTok * 64 * 2;     // 16 KB: 128 tokens x 64 p
  static constexpr int kRowG = 2 * kRowGBox;         // 128 p
  static constexpr int kRowP = kCol * kNR * 2;       // 128 p x K
  static constexpr int kRowStage = kRowG + kRowP;
  static constexpr int kColABox = kTok * 64 * 2;     // 16 KB: 128 tokens x 64 d
  static constexpr int kColA = 2 * kColABox;
  static constexpr int kColWBox = kNC * 64 * 2;      // 2K rows x 64 tokens
  static constexpr int kColW = 2 * kColWBox;
  static constexpr int kColStage = kColA + kColW;
  static constexpr int kRing = kColStages * kColStage;
  static constexpr int kRowSlot = kRing / kRowStages;
  static constexpr int kColSlot = kRing / kColStages;
  static constexpr int kAccR = K < 32 ? 32 : K;
  static constexpr int kColAcc0 = 2 * kAccR;
  static constexpr int kTmemCols = 256;
  static constexpr int kBars = 2 * kRowStages + 2 * kColStages + 8 + 4;  // + exchange
  static constexpr int xchg(int cl) { return cl <= 1 ? 0 : (cl - 1) * (kRows / cl) * K * 4; }
  static constexpr int kCtrl = 1024;  // barriers, TMEM slot, flags, norms
  static constexpr int smem(int cl) { return 1024 + kRing + kCtrl + xchg(cl); }
  static_assert(kRowSlot >= kRowStage && kRowSlot % 1024 == 0, "sketch slot");
  static_assert(kRowStages % kColStages == 0, "projection slots overlay whole sketch slots");
  static_assert(kColSlot % 1024 == 0, "projection slot");
  static_assert(kColAcc0 + 2 * kNC <= kTmemCols, "TMEM columns");
  static_assert(K == 16 || K == 32, "k = 16 or 32");
};

struct Phase {
  int split;          // 1: one block per cluster, units split by rank
  long long nblocks;  // blocks of this phase
  int upb;            // units per block
};

struct HArgs {
  int T, p, d;
  int mtiles;    // sketch blocks per sample
  int nchunks;   // projection blocks per sample
  long long tpad;
  Phase ph1, ph2;
  int ready_target;  // ready[i] value meaning "W_i complete"
  __nv_bfloat16* W;
  int* ready;        // [B]
  int* tickets;      // [B]
  float* chunk_norms;  // [B * nchunks]
  float* n_out;
  int accumulate;
};

// Blocks and units of this CTA in one phase.
struct Mine {
  long long first, step;  // blocks first, first + step, ... < nblocks
  int ulo, uhi;           // units of each block
};

__device__ __forceinline__ Mine mine(const Phase& ph, int cl, int rank) {
  Mine m;
  if (ph.split) {
    m.first = blockIdx.x / cl;
    m.step = gridDim.x / cl;
    m.ulo = rank * ph.upb / cl;
    m.uhi = (rank + 1) * ph.upb / cl;
  } else {
    m.first = blockIdx.x;
    m.step = gridDim.x;
    m.ulo = 0;
    m.uhi = ph.upb;
  }
  return m;
}

__device__ __forceinline__ long long count_blocks(const Phase& ph, const Mine& m) {
  return ph.nblocks > m.first ? (ph.nblocks - 1 - m.first) / m.step + 1 : 0;
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait until *p >= target (acquire); false (error recorded) on timeout.
__device__ __forceinline__ bool wait_geq(const int* p, int target) {
  if (ld_acquire(p) >= target) return true;
  const unsigned long long t0 = globaltimer_ns();
  unsigned ns = 64;
  while (true) {
    __nanosleep(ns);
    if (ld_acquire(p) >= target) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_error(DPRC_DEVERR_READY);
      return false;
    }
    if (ns < 512) ns *= 2;
  }
}

// Cluster exchange state of one CTA.
struct Xchg {
  float* recv;          // [cl-1][128/cl][K] rows sent to this rank
  uint64_t* recv_bar;   // (cl-1) * 128/cl arrivals per round
  uint64_t* free_bar;   // (cl-1) arrivals per round: owners have read our rows
  uint64_t* norm_bar;   // [2] rank 0: cl-1 arrivals per block (by block parity)
  float* norms;         // [2][8] rank 0: per-rank partial norms
};

// Reduce-scatter of one 128-row block of fp32 partials across the cluster
// (round `rnd` of this CTA's exchanges, `last`: no later round).  Each thread
// holds row `row` in y[]; the threads whose row lies in this rank's range
// end with the sum over ranks in rank order and return true.
template <int K>
__device__ __forceinline__ bool xchg_rows(const Xchg& xs, int cl, int rank, int row, int rnd,
                                          bool last, float (&y)[K], bool& ok) {
  const int R = kRows / cl;
  const int owner = row / R;
  const int r_in = row - owner * R;
  bool mine_row = owner == rank;
  if (!mine_row) {
    // the owner must have read our rows of the previous round
    if (rnd > 0 && !mbar_wait(xs.free_bar, static_cast<uint32_t>(rnd - 1) & 1, DPRC_DEVERR_CLUSTER))
      ok = false;
    const int slot = rank < owner ? rank : rank - 1;
    const uint32_t dst = map_to_rank(xs.recv + (static_cast<size_t>(slot) * R + r_in) * K, owner);
#pragma unroll
    for (int c4 = 0; c4 < K / 4; ++c4)
      st_cluster_f4(dst + 16 * c4, make_float4(y[4 * c4], y[4 * c4 + 1], y[4 * c4 + 2], y[4 * c4 + 3]));
    mbar_arrive_remote(map_to_rank(xs.recv_bar, owner));
  } else {
    if (!mbar_wait_cluster(xs.recv_bar, static_cast<uint32_t>(rnd) & 1, DPRC_DEVERR_CLUSTER))
      ok = false;
    float acc[K];
#pragma unroll
    for (int t = 0; t < K; ++t) acc[t] = 0.f;
    for (int s = 0; s < cl; ++s) {
      if (s == rank) {
#pragma unroll
        for (int t = 0; t < K; ++t) acc[t] += y[t];
      } else {
        const int slot = s < rank ? s : s - 1;
        const float4* src =
            reinterpret_cast<const float4*>(xs.recv + (static_cast<size_t>(slot) * R + r_in) * K);
#pragma unroll
        for (int c4 = 0; c4 < K / 4; ++c4) {
          const float4 v = src[c4];
          acc[4 * c4] += v.x;
          acc[4 * c4 + 1] += v.y;
          acc[4 * c4 + 2] += v.z;
          acc[4 * c4 + 3] += v.w;
        }
      }
    }
#pragma unroll
    for (int t = 0; t < K; ++t) y[t] = acc[t];
  }
  // all rows of this round are read: hand the senders their credit
  named_bar_sync(1, 128);
  if (!last && threadIdx.x == 64) {  // first epilogue thread
    for (int s = 0; s < cl; ++s)
      if (s != rank) mbar_arrive_remote(map_to_rank(xs.free_bar, s));
  }
  return mine_row;
}

template <int K>
__global__ void __launch_bounds__(192, 1)
    tc_hutch_kernel(const __grid_constant__ CUtensorMap map_g,
                    const __grid_constant__ CUtensorMap map_p,
                    const __grid_constant__ CUtensorMap map_a,
                    const __grid_constant__ CUtensorMap map_w, const HArgs a, const int cl) {
  using Cfg = HCfg<K>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_red[4];

  uint8_t* ring = align_1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + Cfg::kRing);
  constexpr int RS = Cfg::kRowStages, CS = Cfg::kColStages;
  uint64_t* full_r = bars;              // [RS]
  uint64_t* empty_r = full_r + RS;      // [RS]
  uint64_t* full_c = empty_r + RS;      // [CS]
  uint64_t* empty_c = full_c + CS;      // [CS]
  uint64_t* accf_r = empty_c + CS;      // [2]
  uint64_t* acce_r = accf_r + 2;        // [2]
  uint64_t* accf_c = acce_r + 2;        // [2]
  uint64_t* acce_c = accf_c + 2;        // [2]
  Xchg xs;
  xs.recv_bar = acce_c + 2;
  xs.free_bar = acce_c + 3;
  xs.norm_bar = acce_c + 4;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::kBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  xs.norms = reinterpret_cast<float*>(bars + Cfg::kBars + 2);  // [2][8]
  xs.recv = reinterpret_cast<float*>(ring + Cfg::kRing + Cfg::kCtrl);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a dependent launch (the clip factors) may start now; it waits for this
  // grid's completion before reading anything
  pdl_launch_dependents();
  const int rank = cl > 1 ? static_cast<int>(cluster_ctarank()) : 0;
  const Mine m1 = mine(a.ph1, cl, rank);
  const Mine m2 = mine(a.ph2, cl, rank);
  const long long nb1 = count_blocks(a.ph1, m1);
  const long long nb2 = count_blocks(a.ph2, m2);
  const int nu1 = m1.uhi - m1.ulo;
  const int nu2 = m2.uhi - m2.ulo;

  if (threadIdx.x == 0) {
    for (int s = 0; s < RS; ++s) {
      mbar_init(&full_r[s], 1);
      mbar_init(&empty_r[s], 1);
    }
    for (int s = 0; s < CS; ++s) {
      mbar_init(&full_c[s], 1);
      mbar_init(&empty_c[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&accf_r[s], 1);
      mbar_init(&acce_r[s], 4);
      mbar_init(&accf_c[s], 1);
      mbar_init(&acce_c[s], 4);
      mbar_init(&xs.norm_bar[s], cl > 1 ? cl - 1 : 1);
    }
    if (cl > 1) {
      mbar_init(xs.recv_bar, (cl - 1) * (kRows / cl));
      mbar_init(xs.free_bar, cl - 1);
    }
    fence_mbar_init();
    *abort_flag = 0;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_g);
    tma_prefetch_desc(&map_p);
    tma_prefetch_desc(&map_a);
    tma_prefetch_desc(&map_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cfg::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  if (cl > 1) cluster_sync_all();  // peers' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      bool ok = true;
      long long it1 = 0;
      for (long long j = 0; j < nb1 && ok; ++j) {
        const long long b = m1.first + j * m1.step;
        const int i = static_cast<int>(b / a.mtiles);
        const int t0 = static_cast<int>(b - static_cast<long long>(i) * a.mtiles) * kTok;
        for (int u = m1.ulo; u < m1.uhi; ++u, ++it1) {
          const int s = static_cast<int>(it1 % RS);
          if (!mbar_wait(&empty_r[s], (static_cast<uint32_t>(it1 / RS) & 1) ^ 1,
                         DPRC_DEVERR_PIPE_EMPTY)) {
            ok = false;
            *abort_flag = 1;
            break;
          }
          uint8_t* slot = ring + s * Cfg::kRowSlot;
          mbar_arrive_expect_tx(&full_r[s], Cfg::kRowStage);
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_3d(slot + h * Cfg::kRowGBox, &map_g, &full_r[s], u * kCol + h * 64, t0, i);
          tma_load_3d(slot + Cfg::kRowG, &map_p, &full_r[s], 0, u * kCol, 0);
        }
      }
      // Phase 2.  The A tiles do not depend on phase 1: before waiting for a
      // new sample's sketch, up to CS stages of A are put in flight; otherwise
      // the A and W tiles of a stage go out together.  Two cursors walk the
      // stages (one division per block, not per stage: this thread paces the
      // whole pipeline).
      struct Cursor {
        long long j = 0;  // block index within this CTA's list
        int u = 0, i = 0, ch = 0;
      };
      auto seek = [&](Cursor& c) {
        const long long b = m2.first + c.j * m2.step;
        c.i = static_cast<int>(b / a.nchunks);
        c.ch = static_cast<int>(b - static_cast<long long>(c.i) * a.nchunks);
      };
      auto advance = [&](Cursor& c) {
        if (++c.u == m2.uhi) {
          c.u = m2.ulo;
          ++c.j;
          if (c.j < nb2) seek(c);
        }
      };
      const long long total2 = nb2 * nu2;
      Cursor ca, cw;
      ca.u = cw.u = m2.ulo;
      if (nb2 > 0) {
        seek(ca);
        seek(cw);
      }
      long long it2 = 0, w_ptr = 0;  // stages with A issued / with W issued
      int ready_i = -1;
      while (w_ptr < total2) {
        const bool need_wait = ok && cw.i != ready_i;
        const long long ahead = need_wait ? CS : 1;
        const long long a_to = w_ptr + ahead < total2 ? w_ptr + ahead : total2;
        while (ok && it2 < a_to) {
          const int s = static_cast<int>(it2 % CS);
          if (it2 < CS) {
            // first use of this slot: the sketch slots under it are consumed
            constexpr int kPer = RS / CS;
            for (int q = kPer * s; q < kPer * s + kPer && ok; ++q) {
              const long long uses = it1 > q ? (it1 - 1 - q) / RS + 1 : 0;
              if (uses > 0 && !mbar_wait(&empty_r[q], static_cast<uint32_t>(uses - 1) & 1,
                                         DPRC_DEVERR_PIPE_EMPTY))
                ok = false;
            }
          } else if (!mbar_wait(&empty_c[s], (static_cast<uint32_t>(it2 / CS) & 1) ^ 1,
                                DPRC_DEVERR_PIPE_EMPTY)) {
            ok = false;
          }
          if (!ok) break;
          uint8_t* slot = ring + s * Cfg::kColSlot;
          mbar_arrive_expect_tx(&full_c[s], Cfg::kColStage);
#pragma unroll
          for (int h = 0; h < 2; ++h)
            tma_load_3d(slot + h * Cfg::kColABox, &map_a, &full_c[s], ca.ch * kRows + h * 64,
                        ca.u * kTok, ca.i);
          ++it2;
          advance(ca);
        }
        if (w_ptr >= it2) break;  // nothing left to complete (after an error)
        if (need_wait && ok) {
          if (wait_geq(&a.ready[cw.i], a.ready_target)) {
            fence_proxy_async_global();
            ready_i = cw.i;
          } else {
            ok = false;  // still load W so the issued stages complete; results are void
          }
        }
        const int s = static_cast<int>(w_ptr % CS);
        uint8_t* slot = ring + s * Cfg::kColSlot;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_3d(slot + Cfg::kColA + h * Cfg::kColWBox, &map_w, &full_c[s],
                      cw.u * kTok + h * 64, 0, cw.i);
        ++w_ptr;
        advance(cw);
      }
      if (!ok) *abort_flag = 1;
      // let every copy this thread issued land before the CTA can exit
      for (long long k = it1 - 1; k >= 0 && k >= it1 - RS; --k)
        mbar_wait(&full_r[k % RS], static_cast<uint32_t>(k / RS) & 1, DPRC_DEVERR_PIPE_FULL);
      for (long long k = it2 - 1; k >= 0 && k >= it2 - CS; --k)
        mbar_wait(&full_c[k % CS], static_cast<uint32_t>(k / CS) & 1, DPRC_DEVERR_PIPE_FULL);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      long long it1 = 0;
      constexpr uint32_t idesc1 = make_idesc_bf16(128, Cfg::kNR, false, true);
      constexpr uint32_t p_swz = swz_code_for_bytes(2 * Cfg::kNR);
      for (long long j = 0; j < nb1 && ok; ++j) {
        const int abuf = static_cast<int>(j & 1);
        if (!mbar_wait(&acce_r[abuf], (static_cast<uint32_t>(j >> 1) & 1) ^ 1, DPRC_DEVERR_ACCUM)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int u = 0; u < nu1; ++u, ++it1) {
          const int s = static_cast<int>(it1 % RS);
          if (!mbar_wait(&full_r[s], static_cast<uint32_t>(it1 / RS) & 1, DPRC_DEVERR_PIPE_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t ga = smem_u32(ring + s * Cfg::kRowSlot);
          const uint32_t pa = ga + Cfg::kRowG;
#pragma unroll
          for (int kk = 0; kk < kCol / 16; ++kk) {
            // G tile: two boxes of 128 token rows x 64 p, K-major, 128-byte swizzle.
            const uint64_t ad =
                make_sdesc(ga + (kk >> 2) * Cfg::kRowGBox + (kk & 3) * 32, 16, 1024, kSwz128);
            // P tile: 128 p rows x K columns, MN-major, one swizzle atom wide.
            const uint64_t bd = make_sdesc(pa + kk * 32 * Cfg::kNR, 16, 16 * Cfg::kNR, p_swz);
            umma_bf16(tmem + abuf * Cfg::kAccR, ad, bd, idesc1, (u == 0 && kk == 0) ? 0u : 1u);
          }
          umma_commit(&empty_r[s]);
        }
        if (ok) umma_commit(&accf_r[abuf]);
      }
      long long it2 = 0;
      constexpr uint32_t idesc2 = make_idesc_bf16(128, Cfg::kNC, true, false);
      for (long long j = 0; j < nb2 && ok; ++j) {
        const int abuf = static_cast<int>(j & 1);
        if (!mbar_wait(&acce_c[abuf], (static_cast<uint32_t>(j >> 1) & 1) ^ 1, DPRC_DEVERR_ACCUM)) {
          ok = false;
          break;
        }
        tc_fence_after();
        for (int u = 0; u < nu2; ++u, ++it2) {
          const int s = static_cast<int>(it2 % CS);
          if (!mbar_wait(&full_c[s], static_cast<uint32_t>(it2 / CS) & 1, DPRC_DEVERR_PIPE_FULL)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xa = smem_u32(ring + s * Cfg::kColSlot);
          const uint32_t wa = xa + Cfg::kColA;
#pragma unroll
          for (int kk = 0; kk < kTok / 16; ++kk) {
            // A^T: 128 d (two 64-d atoms, LBO = one box) x 16 tokens (SBO 1 KB).
            const uint64_t ad = make_sdesc(xa + kk * 2048, Cfg::kColABox, 1024, kSwz128);
            // Sketch: 2K rows x 64 tokens per box, K-major, 128-byte swizzle.
            const uint64_t bd =
                make_sdesc(wa + (kk >> 2) * Cfg::kColWBox + (kk & 3) * 32, 16, 1024, kSwz128);
            umma_bf16(tmem + Cfg::kColAcc0 + abuf * Cfg::kNC, ad, bd, idesc2,
                      (u == 0 && kk == 0) ? 0u : 1u);
          }
          umma_commit(&empty_c[s]);
        }
        if (ok) umma_commit(&accf_c[abuf]);
      }
      if (!ok) *abort_flag = 1;
    }
  } else {
    // ---------------- epilogue warps 2..5 ----------------
    const int ew = warp - 2;
    const int q = warp & 3;         // TMEM lane quadrant of this warp
    const int row = q * 32 + lane;  // row of the 128-row tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    bool ok = true;
    int rnd = 0;  // cluster exchange rounds so far
    const int rounds = (a.ph1.split ? static_cast<int>(nb1) : 0) +
                       (a.ph2.split ? static_cast<int>(nb2) : 0);
    // phase 1: sketch rows -> W hi/lo, then count the block done
    for (long long j = 0; j < nb1; ++j) {
      const int abuf = static_cast<int>(j & 1);
      bool live = ok &&
                  mbar_wait(&accf_r[abuf], static_cast<uint32_t>(j >> 1) & 1, DPRC_DEVERR_ACCUM) &&
                  *abort_flag == 0;
      live = __all_sync(0xffffffffu, live);  // keep the warp's TMEM loads convergent
      if (!live) ok = false;
      tc_fence_after();
      float y[K];
#pragma unroll
      for (int t = 0; t < K; ++t) y[t] = 0.f;
      if (live) tmem_ld_cols<K>(tmem + lane_base + abuf * Cfg::kAccR, y);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_r[abuf]);
      bool mine_row = true;
      if (a.ph1.split) {
        mine_row = xchg_rows<K>(xs, cl, rank, row, rnd, rnd + 1 == rounds, y, ok);
        ++rnd;
      }
      const long long b = m1.first + j * m1.step;
      const int i = static_cast<int>(b / a.mtiles);
      const int t = static_cast<int>(b - static_cast<long long>(i) * a.mtiles) * kTok + row;
      if (mine_row && ok && t < a.T) {
        __nv_bfloat16* wi = a.W + static_cast<size_t>(i) * 2 * K * a.tpad + t;
#pragma unroll
        for (int c = 0; c < K; ++c) {
          __nv_bfloat16 hi, lo;
          split_hilo(y[c], hi, lo);
          wi[static_cast<size_t>(c) * a.tpad] = hi;
          wi[static_cast<size_t>(K + c) * a.tpad] = lo;
        }
      }
      fence_proxy_async_global();  // these rows are read by TMA (async proxy)
      named_bar_sync(1, 128);
      if (ew == 0 && lane == 0 && ok) {
        __threadfence();
        atomicAdd(&a.ready[i], 1);
      }
    }
    // phase 2: squared norms of the projection blocks
    for (long long j = 0; j < nb2; ++j) {
      const int abuf = static_cast<int>(j & 1);
      bool live = ok &&
                  mbar_wait(&accf_c[abuf], static_cast<uint32_t>(j >> 1) & 1, DPRC_DEVERR_ACCUM) &&
                  *abort_flag == 0;
      live = __all_sync(0xffffffffu, live);
      if (!live) ok = false;
      tc_fence_after();
      float y[K];
#pragma unroll
      for (int t = 0; t < K; ++t) y[t] = 0.f;
      if (live) {
        const uint32_t tb = tmem + lane_base + Cfg::kColAcc0 + abuf * Cfg::kNC;
        float hi[K], lo[K];
        tmem_ld_cols<K>(tb, hi);
        tmem_ld_cols<K>(tb + K, lo);
#pragma unroll
        for (int t = 0; t < K; ++t) y[t] = hi[t] + lo[t];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_c[abuf]);
      bool mine_row = true;
      if (a.ph2.split) {
        mine_row = xchg_rows<K>(xs, cl, rank, row, rnd, rnd + 1 == rounds, y, ok);
        ++rnd;
      }
      const long long b = m2.first + j * m2.step;
      const int i = static_cast<int>(b / a.nchunks);
      const int ch = static_cast<int>(b - static_cast<long long>(i) * a.nchunks);
      float sq = 0.f;
      if (mine_row && ok && ch * kRows + row < a.d) {
#pragma unroll
        for (int t = 0; t < K; ++t) sq = fmaf(y[t], y[t], sq);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      if (lane == 0) s_red[ew] = sq;
      named_bar_sync(1, 128);
      if (ew == 0 && lane == 0) {
        const float part = (s_red[0] + s_red[1]) + (s_red[2] + s_red[3]);
        float chunk = part;
        bool leader = true;
        if (a.ph2.split) {
          float* nb = xs.norms + (j & 1) * 8;
          if (rank != 0) {
            st_cluster_f32(map_to_rank(nb + rank, 0), part);
            mbar_arrive_remote(map_to_rank(&xs.norm_bar[j & 1], 0));
            leader = false;
          } else {
            if (!mbar_wait_cluster(&xs.norm_bar[j & 1], static_cast<uint32_t>(j >> 1) & 1,
                                   DPRC_DEVERR_CLUSTER))
              ok = false;
            nb[0] = part;
            chunk = 0.f;
            for (int s = 0; s < cl; ++s) chunk += nb[s];
          }
        }
        if (leader && ok) {
          a.chunk_norms[b] = chunk;
          __threadfence();
          const int old = atomicAdd(&a.tickets[i], 1);
          if (old == a.nchunks - 1) {
            // last block of sample i: sum its blocks in order, reset the counters
            __threadfence();
            float sum = 0.f;
            for (int c = 0; c < a.nchunks; ++c)
              sum += __ldcg(&a.chunk_norms[static_cast<size_t>(i) * a.nchunks + c]);
            a.n_out[i] = (a.accumulate ? a.n_out[i] : 0.f) + sum;
            a.tickets[i] = 0;
            a.ready[i] = 0;
          }
        }
      }
      named_bar_sync(1, 128);
    }
  }

  __syncwarp();  // reconverge each warp before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
  if (cl > 1) cluster_sync_all();  // no peer still addresses this CTA's shared memory
}

template <int K>
cudaError_t set_smem_once() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> done[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(tc_hutch_kernel<K>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           HCfg<K>::smem(8));
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDev) done[dev].store(1, std::memory_order_release);
  return e;
}

// CTAs of this kernel that may run at once in one cooperative launch with
// clusters of cl: the driver's occupancy figures (one CTA per SM: the
// tensor-memory kernels are counted as such), cached per device and cl.
template <int K>
int resident_ctas(int cl) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> cache[kMaxDev][4];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return 0;
  const int ci = cl == 1 ? 0 : (cl == 2 ? 1 : (cl == 4 ? 2 : 3));
  int v = cache[dev][ci].load(std::memory_order_acquire);
  if (v > 0) return v;
  const int smem = HCfg<K>::smem(cl);
  if (cl == 1) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_hutch_kernel<K>, 192, smem) !=
        cudaSuccess)
      return 0;
    v = per_sm * device_sm_count();
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl * device_sm_count());
    cfg.blockDim = dim3(192);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = cl;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int ncl = 0;
    if (cudaOccupancyMaxActiveClusters(&ncl, tc_hutch_kernel<K>, &cfg) != cudaSuccess) return 0;
    v = ncl * cl;
  }
  cache[dev][ci].store(v, std::memory_order_release);
  return v;
}

template <int K>
cudaError_t launch_k(const CUtensorMap& mg, const CUtensorMap& mp, const CUtensorMap& ma,
                     const CUtensorMap& mw, const HArgs& a, int grid, int cl, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = HCfg<K>::smem(cl);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeCooperative;
  attr[na].val.cooperative = 1;
  ++na;
  if (cl > 1) {
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = cl;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
  }
  cfg.attrs = attr;
  cfg.numAttrs = na;
  return cudaLaunchKernelEx(&cfg, tc_hutch_kernel<K>, mg, mp, ma, mw, a, cl);
}

// Cluster size a phase of `nblocks` blocks of `upb` units wants on `slots`
// CTAs: 1 when the blocks fill most slots, else the largest power of two
// (<= 8, <= upb) that keeps the split blocks within the slots.
int want_cl(long long nblocks, int upb, int slots) {
  if (nblocks * 4 >= static_cast<long long>(slots) * 3) return 1;
  int cl = 1;
  while (cl < 8 && nblocks * cl * 2 <= slots && cl * 2 <= upb) cl *= 2;
  return cl;
}

}  // namespace

cudaError_t read_device_error_hutch(int32_t* out, bool reset) {
  return read_tu_device_error(out, reset);
}

bool fused_hutch_supported(int64_t k) { return k == 16 || k == 32; }

namespace {

// Devices on which the cooperative launch was refused once keep using the
// two-kernel path.
constexpr int kMaxDevices = 64;
std::atomic<int> g_refused[kMaxDevices];

// Schedule of one fused launch (phases, cluster size, grid); false when the
// kernel cannot run with these sizes on the current device.
bool plan_fused(int64_t B, int64_t T, int64_t d, int64_t p, int64_t k, HArgs& a, int& grid_out,
                int& cl_out) {
  if (!fused_hutch_supported(k)) return false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  if (g_refused[dev].load(std::memory_order_acquire)) return false;
  const int ik = static_cast<int>(k);
  const int slots = device_sm_count();  // one CTA per SM
  a.T = static_cast<int>(T);
  a.p = static_cast<int>(p);
  a.d = static_cast<int>(d);
  a.mtiles = static_cast<int>((T + kTok - 1) / kTok);
  a.nchunks = static_cast<int>((d + kRows - 1) / kRows);
  a.ph1.nblocks = B * a.mtiles;
  a.ph1.upb = static_cast<int>((p + kCol - 1) / kCol);
  a.ph2.nblocks = B * a.nchunks;
  a.ph2.upb = a.mtiles;
  const int cl1 = want_cl(a.ph1.nblocks, a.ph1.upb, slots);
  const int cl2 = want_cl(a.ph2.nblocks, a.ph2.upb, slots);
  const int cl = cl1 > cl2 ? cl1 : cl2;
  if ((ik == 16 ? set_smem_once<16>() : set_smem_once<32>()) != cudaSuccess) return false;
  const int resident = ik == 16 ? resident_ctas<16>(cl) : resident_ctas<32>(cl);
  if (resident < cl) return false;
  a.ph1.split = cl1 > 1 && a.ph1.upb >= cl ? 1 : 0;
  a.ph2.split = cl2 > 1 && a.ph2.upb >= cl ? 1 : 0;
  // Grid: the multiple of cl (up to what is resident) that minimises the
  // bytes the busiest CTA streams in the two phases (a sketch unit is 32 KB of
  // G, a projection unit 32 KB of A); ties go to the smaller grid.
  long long grid = 0, best = -1;
  for (long long ncl = 1; ncl * cl <= resident; ++ncl) {
    const long long g = ncl * cl;
    auto busiest = [&](const Phase& ph, long long unit_bytes) {
      if (ph.split)
        return (ph.nblocks + ncl - 1) / ncl * ((ph.upb + cl - 1) / cl) * unit_bytes;
      return (ph.nblocks + g - 1) / g * ph.upb * unit_bytes;
    };
    const long long cost = busiest(a.ph1, 32) + busiest(a.ph2, 32);
    if (best < 0 || cost < best) {
      best = cost;
      grid = g;
    }
  }
  if (grid < cl) return false;
  a.ready_target = a.mtiles * (a.ph1.split ? cl : 1);
  grid_out = static_cast<int>(grid);
  cl_out = cl;
  return true;
}

}  // namespace

bool fused_hutch_planned(int64_t B, int64_t T, int64_t d, int64_t p, int64_t k) {
  HArgs a;
  int grid = 0, cl = 0;
  return plan_fused(B, T, d, p, k, a, grid, cl);
}

cudaError_t launch_tc_hutch_fused(const void* A, const void* G, const void* P, int64_t B,
                                  int64_t T, int64_t d, int64_t p, int64_t k, void* W,
                                  int64_t tpad, int* ready, int* tickets, float* chunk_norms,
                                  float* n_out, int accumulate, cudaStream_t s, bool* launched) {
  *launched = false;
  HArgs a;
  int grid = 0, cl = 0;
  if (!plan_fused(B, T, d, p, k, a, grid, cl)) return cudaSuccess;
  const int ik = static_cast<int>(k);
  a.tpad = tpad;
  a.W = static_cast<__nv_bfloat16*>(W);
  a.ready = ready;
  a.tickets = tickets;
  a.chunk_norms = chunk_norms;
  a.n_out = n_out;
  a.accumulate = accumulate;

  CUtensorMap mg, mp, ma, mw;
  if (!make_tmap_3d_bf16(&mg, G, p, T, B, p, T * p, 64, kTok, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_3d_bf16(&mp, P, ik, p, 1, ik, p * ik, ik, kCol, 2 * ik))
    return cudaErrorInvalidValue;
  if (!make_tmap_3d_bf16(&ma, A, d, T, B, d, T * d, 64, kTok, 128)) return cudaErrorInvalidValue;
  if (!make_tmap_3d_bf16(&mw, W, T, 2 * ik, B, tpad, 2 * ik * tpad, 64, 2 * ik, 128))
    return cudaErrorInvalidValue;
  const cudaError_t e = ik == 16 ? launch_k<16>(mg, mp, ma, mw, a, grid, cl, s)
                                 : launch_k<32>(mg, mp, ma, mw, a, grid, cl, s);
  if (e == cudaSuccess) {
    *launched = true;
  } else if (e == cudaErrorCooperativeLaunchTooLarge || e == cudaErrorNotSupported ||
             e == cudaErrorInvalidConfiguration || e == cudaErrorInvalidValue) {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices)
      g_refused[dev].store(1, std::memory_order_release);
  }
  return e;
}

}  // namespace dprc
