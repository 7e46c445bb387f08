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
// Work is cut into blocks of 128 output rows (a 128-token tile for the row
// projection, a (sample, 128-row chunk of c) pair for the column projection),
// each the sum over `upb` units (64 columns of c, or 128 tokens).  Two CTAs run
// per SM, each keeping ~64-96 KB of loads in flight - the shape at which plain
// TMA streaming reaches ~6 TB/s on this GPU.  Blocks are assigned either
//   (a) whole, `bpc` per CTA, when there are enough of them, or
//   (b) one block per thread-block cluster of `cl` CTAs, CTA rank r streaming
//       units [r*upb/cl, (r+1)*upb/cl); the fp32 partials are then reduced
//       through distributed shared memory: rank q owns rows [q*128/cl, ...),
//       receives the other ranks' rows of that range and sums them in rank
//       order, so the result does not depend on timing.
// Neither case needs a global cross-CTA reduction, so there is no fix-up tail
// after the last MMA.
//
// Precision: X and R are bf16 (exact in fp32); accumulation is fp32 in TMEM.
// The fp32 sketch W is carried to the second contraction as two bf16 planes
// W = W_hi + W_lo (|W - W_hi - W_lo| <= 2^-17 |W|), multiplied as one MMA of
// width 2n whose two column halves are summed in the epilogue.

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace dprc {

namespace {

constexpr int kRowTile = 128;   // tokens per row-projection tile (MMA M)
constexpr int kTileC = 64;      // c per row-projection unit (128 B of bf16)
constexpr int kColChunk = 128;  // output rows per column-projection block (MMA M)
constexpr int kTileT = 128;     // T rows per column-projection unit

// Block schedule shared by both kernels (see the file comment).
struct Sched {
  int cl;             // CTAs per cluster splitting one block (1, 2, 4 or 8)
  int bpc;            // whole blocks per CTA when cl == 1
  long long nblocks;  // blocks in the launch
  int upb;            // units per block
};

struct CtaWork {
  long long b0, b1;  // blocks [b0, b1)
  int ulo, uhi;      // units [ulo, uhi) of each of them
  int rank;          // rank in the cluster
};

__device__ __forceinline__ CtaWork cta_work(const Sched& s) {
  CtaWork w;
  if (s.cl == 1) {
    w.rank = 0;
    w.b0 = static_cast<long long>(blockIdx.x) * s.bpc;
    w.b1 = w.b0 + s.bpc < s.nblocks ? w.b0 + s.bpc : s.nblocks;
    w.ulo = 0;
    w.uhi = s.upb;
  } else {
    w.rank = static_cast<int>(cluster_ctarank());
    w.b0 = blockIdx.x / s.cl;
    w.b1 = w.b0 + 1;
    w.ulo = w.rank * s.upb / s.cl;
    w.uhi = (w.rank + 1) * s.upb / s.cl;
  }
  return w;
}

// Shared memory of the cluster reduction: receive buffer for the rows this
// rank owns from every other rank, plus two barriers and a small buffer of
// per-rank partial norms (used by rank 0).
struct XchgSmem {
  float* recv;         // [cl-1][128/cl][N] fp32
  uint64_t* recv_bar;  // expects (cl-1) * 128/cl arrivals
  uint64_t* norm_bar;  // rank 0: expects cl-1 arrivals
  float* norms;        // rank 0: [8]
};

template <int N>
__host__ __device__ constexpr int xchg_bytes(int cl) {
  return cl <= 1 ? 0 : (cl - 1) * (128 / cl) * N * 4;
}

// Reduce-scatter of one 128-row block of fp32 partials across the cluster:
// every thread holds row `row` in y[]; afterwards the threads whose row is in
// this rank's range hold the full sum (in rank order) and return true.
template <int N>
__device__ __forceinline__ bool cluster_reduce_rows(const XchgSmem& xs, int cl, int rank, int row,
                                                    float (&y)[N], bool& ok) {
  const int R = 128 / cl;
  const int owner = row / R;
  const int r_in = row - owner * R;
  if (owner != rank) {
    const int slot = rank < owner ? rank : rank - 1;  // sender index at the owner
    if (!DPRC_IN(owner < cl && slot >= 0 && slot < cl - 1 && r_in < R)) return false;
    const uint32_t dst = map_to_rank(xs.recv + (static_cast<size_t>(slot) * R + r_in) * N, owner);
#pragma unroll
    for (int c4 = 0; c4 < N / 4; ++c4)
      st_cluster_f4(dst + 16 * c4, make_float4(y[4 * c4], y[4 * c4 + 1], y[4 * c4 + 2], y[4 * c4 + 3]));
    mbar_arrive_remote(map_to_rank(xs.recv_bar, owner));
    return false;
  }
  if (!mbar_wait_cluster(xs.recv_bar, 0, DPRC_DEVERR_CLUSTER)) ok = false;
  float acc[N];
#pragma unroll
  for (int t = 0; t < N; ++t) acc[t] = 0.f;
  for (int s = 0; s < cl; ++s) {
    if (s == rank) {
#pragma unroll
      for (int t = 0; t < N; ++t) acc[t] += y[t];
    } else {
      const int slot = s < rank ? s : s - 1;
      const float4* src =
          reinterpret_cast<const float4*>(xs.recv + (static_cast<size_t>(slot) * R + r_in) * N);
#pragma unroll
      for (int c4 = 0; c4 < N / 4; ++c4) {
        const float4 v = src[c4];
        acc[4 * c4] += v.x;
        acc[4 * c4 + 1] += v.y;
        acc[4 * c4 + 2] += v.z;
        acc[4 * c4 + 3] += v.w;
      }
    }
  }
#pragma unroll
  for (int t = 0; t < N; ++t) y[t] = acc[t];
  return true;
}

// Shared prologue of both kernels: pipeline barriers, the MMA drain barrier,
// cluster barriers.
template <int kStages>
__device__ __forceinline__ void init_barriers(uint64_t* full, uint64_t* empty, uint64_t* accf,
                                              uint64_t* acce, uint64_t* drain, const XchgSmem& xs,
                                              int cl) {
  for (int s = 0; s < kStages; ++s) {
    mbar_init(&full[s], 1);
    mbar_init(&empty[s], 1);
  }
  for (int b = 0; b < 2; ++b) {
    mbar_init(&accf[b], 1);
    mbar_init(&acce[b], 4);
  }
  mbar_init(drain, 1);
  if (cl > 1) {
    mbar_init(xs.recv_bar, (cl - 1) * (128 / cl));
    mbar_init(xs.norm_bar, cl - 1);
  }
  fence_mbar_init();
}

// ===========================================================================
// Row projection.  Block = 128-token tile; unit = 64 columns of c.
// Warp 0 lane 0: TMA producer.  Warp 1: TMEM allocator, lane 0 issues the
// MMAs.  Warps 2..5: epilogue; warp w owns TMEM lanes 32*(w%4).. = tokens of
// the tile.  The accumulator is double-buffered across blocks.
// ===========================================================================
struct RowArgs {
  int T, c, mtiles;
  Sched sched;
  int r_batched;
  __nv_bfloat16* W;
  long long tpad;
  int* zero_ptr;
  int zero_ints;
  // launched as a programmatic dependent that runs beside the previous
  // kernel (its inputs are older): CTA 0 waits for that kernel to complete
  // before it exits, so this kernel's completion implies the other's (the
  // other CTAs leave as they finish and free their slots)
  int wait_end;
  // if set, ready[i] counts the blocks of sample i whose sketch rows are in
  // memory: after a block's rows, one add with release (the column projection
  // launched after this kernel waits on it instead of this kernel's end)
  int* ready;
};

template <int NMMA, bool HILO_IN>
struct RowCfg {
  static constexpr int kStages = NMMA >= 64 ? 3 : 4;
  static constexpr int kXBytes = kRowTile * kTileC * 2;  // 16 KB
  static constexpr int kRBytes = kTileC * NMMA * 2;      // 2, 4 or 8 KB
  static constexpr int kStageBytes = kXBytes + kRBytes;
  static constexpr int kN = HILO_IN ? NMMA / 2 : NMMA;
  static constexpr int kAcc = NMMA < 32 ? 32 : NMMA;
  static constexpr int kTmemCols = 2 * kAcc;
  static constexpr int kBase = kStages * kStageBytes + 1024 + 256;
  static constexpr int smem(int cl) { return kBase + xchg_bytes<kN>(cl); }
  static_assert(NMMA == 16 || NMMA == 32 || NMMA == 64, "MN-major R atom is one swizzle row");
};

template <int NMMA, bool HILO_IN>
__device__ __forceinline__ void write_sketch_row(__nv_bfloat16* wi, long long tpad,
                                                 const float (&y)[RowCfg<NMMA, HILO_IN>::kN]) {
  constexpr int kN = RowCfg<NMMA, HILO_IN>::kN;
#pragma unroll
  for (int j = 0; j < kN; ++j) {
    __nv_bfloat16 hi, lo;
    split_hilo(y[j], hi, lo);
    wi[static_cast<size_t>(j) * tpad] = hi;
    wi[static_cast<size_t>(kN + j) * tpad] = lo;
  }
}

template <int NMMA, bool HILO_IN>
__global__ void __launch_bounds__(192, 2)
    tc_rowproj_kernel(const __grid_constant__ CUtensorMap map_x,
                      const __grid_constant__ CUtensorMap map_r, const RowArgs a) {
  using Cfg = RowCfg<NMMA, HILO_IN>;
  constexpr int kN = Cfg::kN;
  extern __shared__ uint8_t smem_raw[];

  const Sched& sc = a.sched;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // The schedule splits blocks over clusters of sc.cl CTAs; a launch of any
  // other cluster shape would address ranks that do not exist: refuse it.
  if (cluster_nctarank() != static_cast<uint32_t>(sc.cl)) {
    if (threadIdx.x == 0) record_error(DPRC_DEVERR_LAUNCH);
    return;
  }
  // The whole grid fits at once: the next kernel may start its prologue.
  pdl_launch_dependents();
  if (blockIdx.x == 0 && a.zero_ptr != nullptr)
    for (int z = threadIdx.x; z < a.zero_ints; z += blockDim.x) a.zero_ptr[z] = 0;
  const CtaWork wk = cta_work(sc);
  const int nu = wk.uhi - wk.ulo;

  uint8_t* smem = align_1024(smem_raw);
  uint8_t* sx = smem;
  uint8_t* sr = smem + Cfg::kStages * Cfg::kXBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sr + Cfg::kStages * Cfg::kRBytes);
  uint64_t* empty = full + Cfg::kStages;
  uint64_t* accf = empty + Cfg::kStages;
  uint64_t* acce = accf + 2;
  XchgSmem xs;
  xs.recv_bar = acce + 2;
  xs.norm_bar = acce + 3;
  uint64_t* drain = acce + 4;  // MMA thread: all its MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  xs.norms = reinterpret_cast<float*>(tmem_slot + 2);
  xs.recv = reinterpret_cast<float*>(smem + Cfg::kBase - 1024);

  // the producer (thread 0) issues the first stages right after initialising
  // the barriers, so their DRAM round trip overlaps the TMEM allocation and the
  // CTA barrier
  // X is streamed once per launch (the operand after it in every sequence of
  // this library is the other one): its tiles carry the evict-first L2 policy,
  // so the sketch operand and the outputs keep their place in L2
  auto load_stage = [&](long long it, int s) {
    const long long b = wk.b0 + it / nu;
    const int kc = wk.ulo + static_cast<int>(it % nu);
    const int i = static_cast<int>(b / a.mtiles);
    const int t0 = static_cast<int>(b - static_cast<long long>(i) * a.mtiles) * kRowTile;
    mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
    tma_load_3d_hint(sx + s * Cfg::kXBytes, &map_x, &full[s], kc * kTileC, t0, i,
                     l2_policy_evict_first());
    tma_load_3d(sr + s * Cfg::kRBytes, &map_r, &full[s], 0, kc * kTileC, a.r_batched ? i : 0);
  };
  const long long total_units = wk.b1 > wk.b0 ? (wk.b1 - wk.b0) * nu : 0;
  const int pre = static_cast<int>(total_units < Cfg::kStages ? total_units : Cfg::kStages);
  if (threadIdx.x == 0) {
    init_barriers<Cfg::kStages>(full, empty, accf, acce, drain, xs, sc.cl);
    *abort_flag = 0;
    for (int it = 0; it < pre; ++it) load_stage(it, it);
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
  if (sc.cl > 1) cluster_sync_all();  // peers' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0 && wk.b1 > wk.b0) {
      long long it = 0;
      bool ok = true;
      const uint64_t pol = l2_policy_evict_first();
      for (long long b = wk.b0; b < wk.b1 && ok; ++b) {
        const int i = static_cast<int>(b / a.mtiles);
        const int t0 = static_cast<int>(b - static_cast<long long>(i) * a.mtiles) * kRowTile;
        for (int kc = wk.ulo; kc < wk.uhi; ++kc, ++it) {
          if (it < pre) continue;  // issued before the CTA barrier
          const int s = static_cast<int>(it % Cfg::kStages);
          const uint32_t ph = static_cast<uint32_t>(it / Cfg::kStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, DPRC_DEVERR_PIPE_EMPTY)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
          tma_load_3d_hint(sx + s * Cfg::kXBytes, &map_x, &full[s], kc * kTileC, t0, i, pol);
          tma_load_3d(sr + s * Cfg::kRBytes, &map_r, &full[s], 0, kc * kTileC,
                      a.r_batched ? i : 0);
        }
      }
      // let the copies this thread issued land before the CTA can exit
      for (long long k = it - 1; k >= 0 && k >= it - Cfg::kStages; --k)
        mbar_wait(&full[k % Cfg::kStages], (k / Cfg::kStages) & 1, DPRC_DEVERR_PIPE_FULL);
    }
  } else if (warp == 1) {
    if (lane == 0 && wk.b1 > wk.b0) {
      constexpr uint32_t idesc = make_idesc_bf16(128, NMMA, false, true);
      constexpr uint32_t r_swz = swz_code_for_bytes(2 * NMMA);
      long long it = 0;
      int seg = 0;
      bool ok = true, issued = false;
      for (long long b = wk.b0; b < wk.b1 && ok; ++b, ++seg) {
        const int abuf = seg & 1;
        if (!mbar_wait(&acce[abuf], ((seg >> 1) & 1) ^ 1, DPRC_DEVERR_ACCUM)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        for (int kc = wk.ulo; kc < wk.uhi; ++kc, ++it) {
          const int s = static_cast<int>(it % Cfg::kStages);
          const uint32_t ph = static_cast<uint32_t>(it / Cfg::kStages) & 1;
          if (!mbar_wait(&full[s], ph, DPRC_DEVERR_PIPE_FULL)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xa = smem_u32(sx + s * Cfg::kXBytes);
          const uint32_t ra = smem_u32(sr + s * Cfg::kRBytes);
#pragma unroll
          for (int kk = 0; kk < kTileC / 16; ++kk) {
            // X tile: 128 token rows x 64 c, K-major, 128-byte swizzle.
            const uint64_t ad = make_sdesc(xa + kk * 32, 16, 1024, kSwz128);
            // R tile: 64 c rows x NMMA columns, MN-major, one swizzle atom
            // wide; 8-row atoms of 16*NMMA bytes, a K=16 step is 32*NMMA bytes.
            const uint64_t bd = make_sdesc(ra + kk * 32 * NMMA, 16, 16 * NMMA, r_swz);
            umma_bf16(tmem + abuf * Cfg::kAcc, ad, bd, idesc,
                      (kc == wk.ulo && kk == 0) ? 0u : 1u);
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
    const int q = warp & 3;
    const int row = q * 32 + lane;  // token within the tile = TMEM lane
    bool ok = true;
    int seg = 0;
    for (long long b = wk.b0; b < wk.b1; ++b, ++seg) {
      const int abuf = seg & 1;
      bool live = ok && mbar_wait(&accf[abuf], (seg >> 1) & 1, DPRC_DEVERR_ACCUM) &&
                  *abort_flag == 0;
      live = __all_sync(0xffffffffu, live);  // keep the warp's TMEM loads convergent
      if (!live) ok = false;
      tc_fence_after();
      float y[kN];
#pragma unroll
      for (int t = 0; t < kN; ++t) y[t] = 0.f;
      if (live) {
        float v[NMMA];
        tmem_ld_cols<NMMA>(tmem + (static_cast<uint32_t>(q * 32) << 16) + abuf * Cfg::kAcc, v);
#pragma unroll
        for (int t = 0; t < kN; ++t) y[t] = HILO_IN ? v[t] + v[kN + t] : v[t];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[abuf]);
      bool mine = true;
      if (sc.cl > 1) mine = cluster_reduce_rows<kN>(xs, sc.cl, wk.rank, row, y, ok);
      const int i = static_cast<int>(b / a.mtiles);
      const int t = static_cast<int>(b - static_cast<long long>(i) * a.mtiles) * kRowTile + row;
      if (mine && ok && t < a.T && DPRC_IN(b < sc.nblocks && t < a.tpad))
        write_sketch_row<NMMA, HILO_IN>(a.W + static_cast<size_t>(i) * 2 * kN * a.tpad + t,
                                        a.tpad, y);
      if (a.ready != nullptr) {
        fence_proxy_async_global();  // the rows are read by TMA (async proxy)
        named_bar_sync(1, 128);
        if (ew == 0 && lane == 0 && ok && DPRC_IN(b < sc.nblocks)) {
          __threadfence();
          atomicAdd(&a.ready[i], 1);
        }
      }
    }
    (void)ew;
  }

  __syncwarp();  // reconverge each warp before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
  // every distributed shared memory access of the cluster is complete before
  // any of its CTAs exits
  if (sc.cl > 1) cluster_sync_all();
  if (a.wait_end && blockIdx.x == 0 && threadIdx.x == 0) pdl_wait();
}

// ===========================================================================
// Column projection.  Block = (sample i, 128-row chunk of c); unit = 128 T
// rows.  Stage: two 16 KB boxes of X (128 T x 64 c each; the operand X^T is
// MN-major) and two boxes of the sketch (64 T x 2n rows each, K-major).  The X
// loads of the first stages are issued before waiting on the previous kernel
// (they do not depend on it), so they overlap its tail.
// ===========================================================================
struct ColArgs {
  int T, c, nchunks;
  Sched sched;
  int* sample_tickets;
  float* chunk_norms;
  int mode;
  float* n_out;
  int accumulate;
  int n_head;
  float w_tail;
  float* y_f32;
  __nv_bfloat16* y_hilo;
  int n_split;  // kColprojSplit: columns [0, n_split) to y_hilo, the rest to y_f32
  // kColprojHpp: the QR factors [B][hpp_rcs] and X P fp32 [B][c][16]
  const float* hpp_rc;
  const float* hpp_yp;
  int hpp_rcs;
  // if set, the producer waits for ready[i] >= ready_target (the sketch
  // kernel's per-sample count) instead of the sketch kernel's end; the
  // epilogue still waits for the end before anything it reads or writes.  In
  // the modes with tickets the sample's last block then sets
  // ready[r * ready_stride + i] = 0 for r < ready_rows.
  int* ready;
  int ready_target;
  int ready_rows;
  int ready_stride;
};

// Hutch++ head and tail of one row of d from Y_M = X M (y) and Y_P = X P
// (yp): Y_Q = (y diag(s)) R^-1 by forward substitution (rinv[j] = 0 leaves
// column j out), ||Y_Q||^2 + ||Y_P - Y_Q C||^2 / 16.  f, in shared memory:
// R^T and C^T (so each column's coefficients are 16 contiguous floats, read
// 4 at a time), s, rinv.
constexpr int kHppF = 2 * 256 + 2 * 16;  // floats of f
__device__ __forceinline__ float hpp_row(const float (&y)[16], const float* __restrict__ yp,
                                         const float* f) {
  const float* RT = f;
  const float* CT = f + 256;
  const float* sc = f + 512;
  const float* rinv = f + 528;
  float yq[16];
  float head = 0.f;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    float t = y[j] * sc[j];
    const float4* r4 = reinterpret_cast<const float4*>(RT + j * 16);
#pragma unroll
    for (int q4 = 0; q4 < (j + 3) / 4; ++q4) {
      const float4 c = r4[q4];
      const float cs[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (4 * q4 + u < j) t = fmaf(-yq[4 * q4 + u], cs[u], t);
    }
    yq[j] = t * rinv[j];
    head = fmaf(yq[j], yq[j], head);
  }
  const float4* p4 = reinterpret_cast<const float4*>(yp);
  float tail = 0.f;
#pragma unroll
  for (int l4 = 0; l4 < 4; ++l4) {
    const float4 pv = p4[l4];
    const float ps[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int l = 4 * l4 + u;
      float t = ps[u];
      const float4* c4 = reinterpret_cast<const float4*>(CT + l * 16);
#pragma unroll
      for (int q4 = 0; q4 < 4; ++q4) {
        const float4 c = c4[q4];
        t = fmaf(-yq[4 * q4], c.x, t);
        t = fmaf(-yq[4 * q4 + 1], c.y, t);
        t = fmaf(-yq[4 * q4 + 2], c.z, t);
        t = fmaf(-yq[4 * q4 + 3], c.w, t);
      }
      tail = fmaf(t, t, tail);
    }
  }
  return head + tail * (1.f / 16.f);
}

// Stages sample i's Hutch++ factors (R, s, C from the QR: row-major R, then s,
// then row-major C) into f as hpp_row reads them, by the 128 epilogue threads
// (index et), then 1 / R_jj of the columns kept.
__device__ __forceinline__ void hpp_stage(const float* __restrict__ rc, float* f, int et) {
  for (int e = et; e < 256; e += 128) {
    const int a2 = e >> 4, j = e & 15;
    f[j * 16 + a2] = rc[e];              // R^T
    f[256 + j * 16 + a2] = rc[272 + e];  // C^T
  }
  if (et < 16) f[512 + et] = rc[256 + et];
  named_bar_sync(1, 128);
  if (et < 16) {
    float cn = 0.f;
    for (int a2 = 0; a2 <= et; ++a2) cn = fmaf(f[et * 16 + a2], f[et * 16 + a2], cn);
    const float rjj = f[et * 16 + et];
    f[528 + et] = rjj * rjj > kHppDropTau * kHppDropTau * cn ? 1.f / rjj : 0.f;
  }
  named_bar_sync(1, 128);
}

template <int NMMA>
struct ColCfg {
  static constexpr int kXBoxBytes = kTileT * 64 * 2;   // 128 T rows x 64 c = 16 KB
  static constexpr int kXBytes = 2 * kXBoxBytes;       // 128 c
  static constexpr int kWBoxBytes = NMMA * 64 * 2;     // NMMA rows x 64 T
  static constexpr int kWBytes = 2 * kWBoxBytes;       // 128 T
  static constexpr int kStageBytes = kXBytes + kWBytes;
  static constexpr int kStages = NMMA >= 128 ? 3 : 2;
  static constexpr int kCtasPerSm = NMMA >= 128 ? 1 : 2;
  // registers per thread: at most what kCtasPerSm CTAs leave of the SM's
  // 64 K, and for NMMA = 32 (the Hutch++ passes beside the QR) few enough
  // that two CTAs fit next to a QR CTA (256 threads x 96 registers)
  static constexpr int kMaxRegs = NMMA >= 128 ? 255 : (NMMA == 64 ? 168 : 104);
  static constexpr int kN = NMMA / 2;
  static constexpr int kAcc = NMMA;
  static constexpr int kTmemCols = 2 * kAcc;
  static constexpr int kBase = kStages * kStageBytes + 1024 + 256;
  static constexpr int smem(int cl) { return kBase + xchg_bytes<kN>(cl); }
  static_assert(kTmemCols * kCtasPerSm <= 512, "TMEM has 512 columns");
};

template <int NMMA>
__global__ void __launch_bounds__(192) __maxnreg__(ColCfg<NMMA>::kMaxRegs)
    tc_colproj_kernel(const __grid_constant__ CUtensorMap map_x,
                      const __grid_constant__ CUtensorMap map_w, const ColArgs a) {
  using Cfg = ColCfg<NMMA>;
  constexpr int kN = Cfg::kN;
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_red[4];
  __shared__ __align__(16) float s_hf[kN == 16 ? kHppF : 4];  // Hutch++ factors (kColprojHpp)

  const Sched& sc = a.sched;
  // The schedule splits blocks over clusters of sc.cl CTAs; a launch of any
  // other cluster shape would address ranks that do not exist: refuse it.
  if (cluster_nctarank() != static_cast<uint32_t>(sc.cl)) {
    if (threadIdx.x == 0) record_error(DPRC_DEVERR_LAUNCH);
    return;
  }
  const CtaWork wk = cta_work(sc);
  const int nu = wk.uhi - wk.ulo;

  uint8_t* smem = align_1024(smem_raw);
  uint8_t* sx = smem;
  uint8_t* sw = smem + Cfg::kStages * Cfg::kXBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sw + Cfg::kStages * Cfg::kWBytes);
  uint64_t* empty = full + Cfg::kStages;
  uint64_t* accf = empty + Cfg::kStages;  // [2]
  uint64_t* acce = accf + 2;              // [2]
  XchgSmem xs;
  xs.recv_bar = acce + 2;
  xs.norm_bar = acce + 3;
  uint64_t* drain = acce + 4;  // MMA thread: all its MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 5);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  xs.norms = reinterpret_cast<float*>(tmem_slot + 2);
  xs.recv = reinterpret_cast<float*>(smem + Cfg::kBase - 1024);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long total = (wk.b1 - wk.b0) * nu;  // units of this CTA
  auto unit = [&](long long it, int& i, int& ch, int& kt) {
    const long long b = wk.b0 + it / nu;
    kt = wk.ulo + static_cast<int>(it % nu);
    i = static_cast<int>(b / a.nchunks);
    ch = static_cast<int>(b - static_cast<long long>(i) * a.nchunks);
  };
  // X is streamed with the evict-first L2 policy when this projection ends the
  // sequence (the norm modes), so the sketch W keeps its place in L2; a
  // projection whose output feeds a next Hutch++ pass leaves X at the default,
  // since that pass starts by reading X again and finds its latest part in L2
  const bool x_last = a.mode == kColprojNorm || a.mode == kColprojHpp;
  auto copy_x = [&](int s, int h, int c0, int c1, int i, uint64_t pol) {
    uint8_t* dst = sx + s * Cfg::kXBytes + h * Cfg::kXBoxBytes;
    if (x_last)
      tma_load_3d_hint(dst, &map_x, &full[s], c0, c1, i, pol);
    else
      tma_load_3d(dst, &map_x, &full[s], c0, c1, i);
  };
  auto load_x = [&](long long it, int s) {
    int i, ch, kt;
    unit(it, i, ch, kt);
    const uint64_t pol = l2_policy_evict_first();
#pragma unroll
    for (int h = 0; h < 2; ++h) copy_x(s, h, ch * kColChunk + h * 64, kt * kTileT, i, pol);
  };
  const int pre = static_cast<int>(total < Cfg::kStages ? total : Cfg::kStages);

  if (threadIdx.x == 0) {
    init_barriers<Cfg::kStages>(full, empty, accf, acce, drain, xs, sc.cl);
    *abort_flag = 0;
    // the producer (this thread) issues the X boxes of the first stages now:
    // X does not depend on the previous kernel, and their DRAM round trip
    // overlaps the TMEM allocation and the CTA barrier
    for (int it = 0; it < pre; ++it) {
      mbar_arrive_expect_tx(&full[it], Cfg::kStageBytes);
      load_x(it, it);
    }
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
  // the peers' barriers must exist before this CTA's first remote arrive,
  // which comes only in the epilogue: arrive now, wait there
  if (sc.cl > 1) cluster_arrive();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0 && total > 0) {
      auto load_w = [&](long long it, int s) {
        int i, ch, kt;
        unit(it, i, ch, kt);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_3d(sw + s * Cfg::kWBytes + h * Cfg::kWBoxBytes, &map_w, &full[s],
                      kt * kTileT + h * 64, 0, i);
      };
      // the sketch is written by the previous kernel: wait for its end, or
      // for each sample's count before the sample's first W tile
      int ready_i = -1;
      bool ready_ok = true;
      auto await_w = [&](int i) {
        if (a.ready == nullptr || i == ready_i || !ready_ok) return;
        if (DPRC_IN(i >= 0 && i < a.ready_stride) &&
            wait_geq(&a.ready[i], a.ready_target, kWaitLimitNs, abort_flag)) {
          fence_proxy_async_global();
        } else {
          ready_ok = false;  // W is still loaded so the issued stages complete; results are void
          *abort_flag = 1;
        }
        ready_i = i;
      };
      if (a.ready == nullptr) pdl_wait();
      for (int it = 0; it < pre; ++it) {
        int i, ch, kt;
        unit(it, i, ch, kt);
        await_w(i);
        load_w(it, it);
      }
      long long issued = pre;
      const uint64_t pol = l2_policy_evict_first();
      // the unit of stage `it` by an incremental cursor (one division per
      // block, none per stage: this thread paces the pipeline)
      int ci, cch, ckt;
      if (pre < total) unit(pre, ci, cch, ckt);
      long long cb = wk.b0 + pre / nu;
      for (long long it = pre; it < total; ++it) {
        const int s = static_cast<int>(it % Cfg::kStages);
        const uint32_t ph = static_cast<uint32_t>(it / Cfg::kStages) & 1;
        if (!mbar_wait(&empty[s], ph ^ 1, DPRC_DEVERR_PIPE_EMPTY)) {
          *abort_flag = 1;
          break;
        }
        mbar_arrive_expect_tx(&full[s], Cfg::kStageBytes);
#pragma unroll
        for (int h = 0; h < 2; ++h) copy_x(s, h, cch * kColChunk + h * 64, ckt * kTileT, ci, pol);
        await_w(ci);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_3d(sw + s * Cfg::kWBytes + h * Cfg::kWBoxBytes, &map_w, &full[s],
                      ckt * kTileT + h * 64, 0, ci);
        ++issued;
        if (++ckt == wk.uhi) {
          ckt = wk.ulo;
          ++cb;
          ci = static_cast<int>(cb / a.nchunks);
          cch = static_cast<int>(cb - static_cast<long long>(ci) * a.nchunks);
        }
      }
      for (long long k = issued - 1; k >= 0 && k >= issued - Cfg::kStages; --k)
        mbar_wait(&full[k % Cfg::kStages], (k / Cfg::kStages) & 1, DPRC_DEVERR_PIPE_FULL);
    }
  } else if (warp == 1) {
    if (lane == 0 && total > 0) {
      constexpr uint32_t idesc = make_idesc_bf16(128, NMMA, true, false);
      long long it = 0;
      int seg = 0;
      bool ok = true, issued = false;
      for (long long b = wk.b0; b < wk.b1 && ok; ++b, ++seg) {
        const int abuf = seg & 1;
        if (!mbar_wait(&acce[abuf], ((seg >> 1) & 1) ^ 1, DPRC_DEVERR_ACCUM)) {
          *abort_flag = 1;
          break;
        }
        tc_fence_after();
        for (int u = 0; u < nu; ++u, ++it) {
          const int s = static_cast<int>(it % Cfg::kStages);
          const uint32_t ph = static_cast<uint32_t>(it / Cfg::kStages) & 1;
          if (!mbar_wait(&full[s], ph, DPRC_DEVERR_PIPE_FULL)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t xa = smem_u32(sx + s * Cfg::kXBytes);
          const uint32_t wa = smem_u32(sw + s * Cfg::kWBytes);
#pragma unroll
          for (int kk = 0; kk < kTileT / 16; ++kk) {
            // X^T: 128 c (two 64-c atoms, LBO = one box) x 16 T (two 8-row
            // atoms, SBO = 1 KB); a K=16 step is 16 rows of 128 B.
            const uint64_t ad = make_sdesc(xa + kk * 2048, Cfg::kXBoxBytes, 1024, kSwz128);
            // Sketch: NMMA rows x 64 T per box, K-major, 128-byte swizzle.
            const uint64_t bd =
                make_sdesc(wa + (kk >> 2) * Cfg::kWBoxBytes + (kk & 3) * 32, 16, 1024, kSwz128);
            umma_bf16(tmem + abuf * Cfg::kAcc, ad, bd, idesc, (u == 0 && kk == 0) ? 0u : 1u);
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
    pdl_wait();  // the sample tickets are cleared by the previous kernel
    if (sc.cl > 1) cluster_wait();
    const int ew = warp - 2;
    const int q = warp & 3;
    const int row = q * 32 + lane;  // row of the 128-row chunk = TMEM lane
    bool ok = true;
    int seg = 0;
    int hpp_i = -1;  // sample whose Hutch++ factors s_hf holds
    if constexpr (kN == 16) {
      // the factors do not depend on this kernel's accumulators: the first
      // block's are staged while its tiles stream
      if (a.mode == kColprojHpp && wk.b0 < wk.b1) {
        hpp_i = static_cast<int>(wk.b0 / a.nchunks);
        hpp_stage(a.hpp_rc + static_cast<size_t>(hpp_i) * a.hpp_rcs, s_hf, threadIdx.x - 64);
      }
    }
    for (long long b = wk.b0; b < wk.b1; ++b, ++seg) {
      const int abuf = seg & 1;
      bool live = ok && mbar_wait(&accf[abuf], (seg >> 1) & 1, DPRC_DEVERR_ACCUM) &&
                  *abort_flag == 0;
      live = __all_sync(0xffffffffu, live);  // keep the warp's TMEM loads convergent
      if (!live) ok = false;
      tc_fence_after();
      float y[kN];
#pragma unroll
      for (int t = 0; t < kN; ++t) y[t] = 0.f;
      if (live) {
        const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + abuf * Cfg::kAcc;
        float hi[kN], lo[kN];
        tmem_ld_cols<kN>(tb, hi);
        tmem_ld_cols<kN>(tb + kN, lo);
#pragma unroll
        for (int t = 0; t < kN; ++t) y[t] = hi[t] + lo[t];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[abuf]);
      bool mine = true;
      if (sc.cl > 1) mine = cluster_reduce_rows<kN>(xs, sc.cl, wk.rank, row, y, ok);
      const int i = static_cast<int>(b / a.nchunks);
      const int ch = static_cast<int>(b - static_cast<long long>(i) * a.nchunks);
      const int grow = ch * kColChunk + row;
      if (a.mode == kColprojNorm || a.mode == kColprojHpp) {
        // this CTA's rows: weighted squares (or the Hutch++ head and tail),
        // then a fixed-order reduction
        float sq = 0.f;
        if (a.mode == kColprojHpp) {
          if constexpr (kN == 16) {
            if (i != hpp_i) {  // a block of the next sample: its factors
              named_bar_sync(1, 128);  // every thread is done with the last ones
              hpp_i = i;
              hpp_stage(a.hpp_rc + static_cast<size_t>(i) * a.hpp_rcs, s_hf, threadIdx.x - 64);
            }
            if (mine && ok && grow < a.c && DPRC_IN(b < sc.nblocks))
              sq = hpp_row(y, a.hpp_yp + (static_cast<size_t>(i) * a.c + grow) * 16, s_hf);
          }
        } else if (mine && ok && grow < a.c) {
#pragma unroll
          for (int t = 0; t < kN; ++t) sq += (t < a.n_head ? 1.f : a.w_tail) * y[t] * y[t];
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
        if (lane == 0) s_red[ew] = sq;
        named_bar_sync(1, 128);
        if (ew == 0) {
          // warp 2: lane 0 gathers the chunk's norm; the whole warp sums a
          // finished sample's chunks (one L2 line per lane, fixed order)
          const float part = (s_red[0] + s_red[1]) + (s_red[2] + s_red[3]);
          float chunk = part;
          int leader = 1;
          if (lane == 0 && sc.cl > 1) {
            if (wk.rank != 0) {
              if (DPRC_IN(wk.rank < 8)) {
                st_cluster_f32(map_to_rank(xs.norms + wk.rank, 0), part);
                mbar_arrive_remote(map_to_rank(xs.norm_bar, 0));
              }
              leader = 0;
            } else {
              if (!mbar_wait_cluster(xs.norm_bar, 0, DPRC_DEVERR_CLUSTER)) ok = false;
              xs.norms[0] = part;
              chunk = 0.f;
              for (int s = 0; s < sc.cl; ++s) chunk += xs.norms[s];
            }
          }
          leader = __shfl_sync(0xffffffffu, leader, 0);
          const bool lok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
          if (!lok) ok = false;
          if (leader && lok && DPRC_IN(b < sc.nblocks)) {
            int last = 0;
            if (lane == 0) {
              a.chunk_norms[b] = chunk;
              __threadfence();
              last = atomicAdd(&a.sample_tickets[i], 1) == a.nchunks - 1;
            }
            if (__shfl_sync(0xffffffffu, last, 0)) {
              __threadfence();
              float sum = 0.f;
              for (int c2 = lane; c2 < a.nchunks; c2 += 32)
                sum += __ldcg(&a.chunk_norms[static_cast<size_t>(i) * a.nchunks + c2]);
#pragma unroll
              for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
              if (lane == 0) {
                a.n_out[i] = (a.accumulate ? a.n_out[i] : 0.f) + sum;
                a.sample_tickets[i] = 0;
                // every block of the sample is past its wait on the count
                // (and those of earlier launches that share the block of counts)
                if (a.ready != nullptr)
                  for (int r = 0; r < a.ready_rows; ++r) a.ready[r * a.ready_stride + i] = 0;
              }
            }
          }
        }
        named_bar_sync(1, 128);
      } else if (mine && ok && grow < a.c && DPRC_IN(b < sc.nblocks)) {
        const size_t yrow = static_cast<size_t>(i) * a.c + grow;
        if (a.mode == kColprojF32 || a.mode == kColprojF32Hilo) {
          float4* d4 = reinterpret_cast<float4*>(a.y_f32 + yrow * kN);
#pragma unroll
          for (int c4 = 0; c4 < kN / 4; ++c4)
            d4[c4] = make_float4(y[4 * c4], y[4 * c4 + 1], y[4 * c4 + 2], y[4 * c4 + 3]);
        }
        if (a.mode == kColprojHilo || a.mode == kColprojF32Hilo)
          store_hilo_row<kN>(a.y_hilo + yrow * 2 * kN, y);
        if (a.mode == kColprojSplit) {
          // the first half as hi/lo rows of kN values, the second as fp32 rows
          constexpr int kH = kN / 2;
          float yh[kH];
#pragma unroll
          for (int t = 0; t < kH; ++t) yh[t] = y[t];
          store_hilo_row<kH>(a.y_hilo + yrow * 2 * kH, yh);
          float4* f4 = reinterpret_cast<float4*>(a.y_f32 + yrow * kH);
#pragma unroll
          for (int c4 = 0; c4 < kH / 4; ++c4)
            f4[c4] = make_float4(y[kH + 4 * c4], y[kH + 4 * c4 + 1], y[kH + 4 * c4 + 2],
                                 y[kH + 4 * c4 + 3]);
        }
      }
    }
  }

  __syncwarp();  // reconverge each warp before the CTA barrier
  if (sc.cl > 1 && warp < 2) cluster_wait();  // the epilogue waited before its first remote access
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, Cfg::kTmemCols);
  }
  // every distributed shared memory access of the cluster is complete before
  // any of its CTAs exits
  if (sc.cl > 1) cluster_sync_all();
}

// Raises a kernel's dynamic shared memory limit once per device (the attribute
// is per context; setting it on every launch costs host time).  Keyed by the
// kernel itself: instantiations share a type, not an attribute.
template <auto Kernel>
cudaError_t set_smem_once(int bytes) {
  constexpr int kMaxDev = 64;
  static std::atomic<int> done[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev && done[dev].load(std::memory_order_acquire) >= bytes)
    return cudaSuccess;
  e = cudaFuncSetAttribute(Kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDev) done[dev].store(bytes, std::memory_order_release);
  return e;
}

template <auto Kernel, typename Args>
cudaError_t launch_sched(int grid, int cl, int smem, int smem_max, bool pdl, cudaStream_t s,
                         const CUtensorMap& m0, const CUtensorMap& m1, const Args& args) {
  cudaError_t e = set_smem_once<Kernel>(smem_max);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int na = 0;
  attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[na].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
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
  return cudaLaunchKernelEx(&cfg, Kernel, m0, m1, args);
}

Sched to_sched(const BlockSched& b) {
  Sched s;
  s.cl = b.cl;
  s.bpc = b.bpc;
  s.nblocks = b.nblocks;
  s.upb = b.upb;
  return s;
}

}  // namespace

int rowproj_ctas_per_sm() { return 2; }
int colproj_ctas_per_sm(int nmma) { return nmma >= 128 ? 1 : 2; }
int colproj_stage_chunk() { return kColChunk; }
int colproj_tile_t() { return kTileT; }

cudaError_t read_device_error_proj(int32_t* out, bool reset) {
  return read_tu_device_error(out, reset);
}

cudaError_t launch_tc_rowproj(const void* X, int64_t B, int64_t T, int64_t c, const void* R,
                              bool r_batched, int nmma, bool hilo_in, void* W, int64_t tpad,
                              const BlockSched& bs, int* zero_ptr, size_t zero_ints,
                              cudaStream_t s, bool beside_previous, int* ready) {
  CUtensorMap mx, mr;
  if (!make_tmap_3d_bf16(&mx, X, c, T, B, c, T * c, kTileC, kRowTile, 128))
    return cudaErrorInvalidValue;
  if (!make_tmap_3d_bf16(&mr, R, nmma, c, r_batched ? B : 1, nmma, c * nmma, nmma, kTileC,
                         2 * nmma))
    return cudaErrorInvalidValue;
  RowArgs a;
  a.T = static_cast<int>(T);
  a.c = static_cast<int>(c);
  a.mtiles = static_cast<int>((T + kRowTile - 1) / kRowTile);
  a.sched = to_sched(bs);
  a.r_batched = r_batched ? 1 : 0;
  a.W = static_cast<__nv_bfloat16*>(W);
  a.tpad = tpad;
  a.zero_ptr = zero_ptr;
  a.zero_ints = static_cast<int>(zero_ints);
  a.wait_end = beside_previous ? 1 : 0;
  a.ready = ready;
#define DPRC_ROW(NM, HL)                                                              \
  if (nmma == NM && hilo_in == HL)                                                    \
    return launch_sched<tc_rowproj_kernel<NM, HL>>(                                   \
        bs.grid, bs.cl, RowCfg<NM, HL>::smem(bs.cl), RowCfg<NM, HL>::smem(8),         \
        beside_previous, s, mx, mr, a);
  DPRC_ROW(16, false)
  DPRC_ROW(32, false)
  DPRC_ROW(64, false)
  DPRC_ROW(32, true)
  DPRC_ROW(64, true)
#undef DPRC_ROW
  return cudaErrorInvalidValue;
}

cudaError_t launch_tc_colproj(const void* X, int64_t B, int64_t T, int64_t c, const void* W,
                              int64_t tpad, int n, const BlockSched& bs, int* sample_tickets,
                              float* chunk_norms, ColprojMode mode, float* n_out, int accumulate,
                              int n_head, float w_tail, float* y_f32, void* y_hilo, bool pdl,
                              cudaStream_t s, int n_split, const float* hpp_rc,
                              const float* hpp_yp, int* ready, int ready_target,
                              int ready_rows) {
  const int nmma = 2 * n;
  if (ready_rows > 0 && mode != kColprojNorm && mode != kColprojHpp)
    return cudaErrorInvalidValue;
  if (mode == kColprojSplit && 2 * n_split != n) return cudaErrorInvalidValue;
  if (mode == kColprojHpp && (n != 16 || hpp_rc == nullptr || hpp_yp == nullptr))
    return cudaErrorInvalidValue;
  CUtensorMap mx, mw;
  if (!make_tmap_3d_bf16(&mx, X, c, T, B, c, T * c, 64, kTileT, 128))
    return cudaErrorInvalidValue;
  if (!make_tmap_3d_bf16(&mw, W, T, nmma, B, tpad, nmma * tpad, 64, nmma, 128))
    return cudaErrorInvalidValue;
  ColArgs a;
  a.T = static_cast<int>(T);
  a.c = static_cast<int>(c);
  a.nchunks = static_cast<int>((c + kColChunk - 1) / kColChunk);
  a.sched = to_sched(bs);
  a.sample_tickets = sample_tickets;
  a.chunk_norms = chunk_norms;
  a.mode = mode;
  a.n_out = n_out;
  a.accumulate = accumulate;
  a.n_head = n_head;
  a.w_tail = w_tail;
  a.y_f32 = y_f32;
  a.y_hilo = static_cast<__nv_bfloat16*>(y_hilo);
  a.n_split = n_split;
  a.hpp_rc = hpp_rc;
  a.hpp_yp = hpp_yp;
  a.hpp_rcs = qr_factor_floats();
  a.ready = ready;
  a.ready_target = ready_target;
  a.ready_rows = ready_rows;
  a.ready_stride = static_cast<int>(B);
#define DPRC_COL(NM)                                                                        \
  if (nmma == NM)                                                                           \
    return launch_sched<tc_colproj_kernel<NM>>(bs.grid, bs.cl, ColCfg<NM>::smem(bs.cl),     \
                                               ColCfg<NM>::smem(8), pdl, s, mx, mw, a);
  DPRC_COL(32)
  DPRC_COL(64)
  DPRC_COL(128)
#undef DPRC_COL
  return cudaErrorInvalidValue;
}

}  // namespace dprc
