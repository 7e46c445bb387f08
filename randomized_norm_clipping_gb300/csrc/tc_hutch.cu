// Hutchinson estimates of one or many layers in one launch, on tensor cores:
//
//   n_i (+)= sum_l || A_l,i^T (G_l,i P_l) ||_F^2
//
// ("Efficient DP-SGD for LLMs with Randomized Clipping", papernotes.org,
// "Key design > Hutchinson": the sketch G P first, then Y = A^T (G P), then
// its squared Frobenius norm; "Overall framework": the layerwise sum).
//
// Each layer is two contractions (those of tc_proj.cu): the sketch
// W_i = G_i P and the projection Y_i = A_i^T W_i.  One persistent kernel,
// every CTA resident at once, runs them as phases:
//
//   phase 1 (sketch)      CTAs take blocks of 128 tokens of one sample and write
//                         W_i as bf16 hi/lo planes; each block then adds one to
//                         the counter ready[l][i] (release);
//   phase 2 (projection)  CTAs take blocks (sample i, 128 rows of d); the TMA
//                         producer issues the A tiles at once, waits until
//                         ready[l][i] is complete (acquire), then loads W; the
//                         epilogue squares Y and a per-(layer, sample) ticket
//                         sums the blocks in order.
//
// With several layers a CTA runs the sketch of layer l + 1 before the
// projection of layer l (S0, S1, P0, S2, P1, ...; phase_at), so by the time
// it projects layer l the other CTAs have long written that layer's sketch,
// and one layer's start-up and tail overlap its neighbours' streaming.  The
// sketch has three buffers: before phase 1 of layer l writes buffer l % 3, it
// waits until every projection block of layer l - 3 (the previous user of
// that buffer) has finished.  Per-layer results go to n_l[l][i]; the last
// layer to finish sample i adds them in layer order (deterministic) into n_i.
//
// The cross-CTA waits are safe because every CTA is resident (the grid is at
// most what fits on the device at once) and every wait is on work that comes
// earlier in the one order all CTAs follow (phase_at).  Every wait is bounded (2 s, or the
// limit a test gives) and records a code in the device error word when it
// runs out; the CTA's other roles then stop at their next wait, the MMA
// thread waits for the MMAs it issued and the producer for its copies, and
// the CTA frees its tensor memory and returns.
//
// Each phase assigns blocks either whole, strided over the CTAs, or one at a
// time to a thread-block cluster whose CTAs split the block's units and
// reduce the fp32 partials through distributed shared memory (credits make
// the receive buffer reusable across blocks, phases and layers).
//
// Counters (ready, tickets, per-sample layer tickets, per-layer projection
// counts) are reset by their last user, so they are zero after every call that
// ends without a device error, and must be zero before the first.
//
// One CTA per SM (the 192 KB ring leaves room for no second one).  The
// shared-memory ring has 4
// slots of 48 KB used by both phases: a sketch stage is 128 tokens x 128 p of
// G (two TMA boxes, 256 contiguous bytes per row) plus 128 rows of P; a
// projection stage 128 tokens x 128 d of A plus the matching 128 tokens of the
// sketch.  TMEM: sketch accumulators (2 x 32 columns) and projection
// accumulators (2 x 2k columns), 256 columns.  Per-layer tensor maps travel as
// kernel parameters (at most kMaxLayers per launch; more layers take several
// launches that accumulate).

#include <atomic>

#include "common.cuh"
#include "internal.h"

namespace dprc {

namespace {

constexpr int kTok = 128;   // tokens per sketch block; tokens per projection unit
constexpr int kCol = 128;   // columns of p per sketch unit (two 64-column boxes)
constexpr int kRows = 128;  // rows of d per projection block
constexpr int kStages = 4;  // ring slots

template <int K>
struct HCfg {
  static constexpr int kNR = K;       // sketch MMA N
  static constexpr int kNC = 2 * K;   // projection MMA N (hi | lo)
  static constexpr int kRowGBox = kTok * 64 * 2;     // 16 KB: 128 tokens x 64 p
  static constexpr int kRowG = 2 * kRowGBox;         // 128 p
  static constexpr int kRowP = kCol * kNR * 2;       // 128 p x K
  static constexpr int kRowStage = kRowG + kRowP;
  static constexpr int kColABox = kTok * 64 * 2;     // 16 KB: 128 tokens x 64 d
  static constexpr int kColA = 2 * kColABox;
  static constexpr int kColWBox = kNC * 64 * 2;      // 2K rows x 64 tokens
  static constexpr int kColW = 2 * kColWBox;
  static constexpr int kColStage = kColA + kColW;
  static constexpr int kSlot = kColStage > kRowStage ? kColStage : kRowStage;
  static constexpr int kRing = kStages * kSlot;
  static constexpr int kAccR = K < 32 ? 32 : K;
  static constexpr int kColAcc0 = 2 * kAccR;
  static constexpr int kTmemCols = 256;
  static constexpr int kBars = 2 * kStages + 8 + 1 + 4;  // ring, accumulators, drain, exchange
  static constexpr int xchg(int cl) { return cl <= 1 ? 0 : (cl - 1) * (kRows / cl) * K * 4; }
  static constexpr int kCtrl = 1024;  // barriers, TMEM slot, flags, norms
  static constexpr int smem(int cl) { return 1024 + kRing + kCtrl + xchg(cl); }
  static_assert(kSlot % 1024 == 0, "slots keep the 1024-byte alignment of swizzled tiles");
  static_assert(kColAcc0 + 2 * kNC <= kTmemCols, "TMEM columns");
  static_assert(K == 16 || K == 32, "k = 16 or 32");
};

struct Phase {
  int split;          // 1: one block per cluster, units split by rank
  long long nblocks;  // blocks of this phase
  int upb;            // units per block
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

// Sketch unit of the u-th stage of a block: the CTA's units [ulo, uhi) in an
// order rotated by the CTA index, so that CTAs streaming at the same moment
// read different 256-byte column ranges of their rows of G (a different
// column range of a row lives in other HBM channels).  The sum over the
// block's units is the same; only its order differs (fixed per CTA).
__device__ __forceinline__ int rot_unit(const Mine& m, int u) {
  const int n = m.uhi - m.ulo;
  const int r = static_cast<int>(blockIdx.x % static_cast<unsigned>(n));
  const int v = u - m.ulo + r;
  return m.ulo + (v >= n ? v - n : v);
}

__device__ __forceinline__ long long count_blocks(const Phase& ph, const Mine& m) {
  return ph.nblocks > m.first ? (ph.nblocks - 1 - m.first) / m.step + 1 : 0;
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
                                          bool last, float (&y)[K], bool& ok,
                                          unsigned long long limit_ns) {
  const int R = kRows / cl;
  const int owner = row / R;
  const int r_in = row - owner * R;
  bool mine_row = owner == rank;
  if (!mine_row) {
    // the owner must have read our rows of the previous round
    if (rnd > 0 && !mbar_wait_lim(xs.free_bar, static_cast<uint32_t>(rnd - 1) & 1,
                                  DPRC_DEVERR_CLUSTER, limit_ns, nullptr))
      ok = false;
    const int slot = rank < owner ? rank : rank - 1;
    if (DPRC_IN(owner < cl && slot >= 0 && slot < cl - 1 && r_in < R)) {
      const uint32_t dst =
          map_to_rank(xs.recv + (static_cast<size_t>(slot) * R + r_in) * K, owner);
#pragma unroll
      for (int c4 = 0; c4 < K / 4; ++c4)
        st_cluster_f4(dst + 16 * c4,
                      make_float4(y[4 * c4], y[4 * c4 + 1], y[4 * c4 + 2], y[4 * c4 + 3]));
      mbar_arrive_remote(map_to_rank(xs.recv_bar, owner));
    }
  } else {
    if (!mbar_wait_cluster(xs.recv_bar, static_cast<uint32_t>(rnd) & 1, DPRC_DEVERR_CLUSTER,
                           limit_ns))
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
        if (!DPRC_IN(slot >= 0 && slot < cl - 1 && r_in < R)) continue;
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
      if (s != rank && DPRC_IN(cl <= 8)) mbar_arrive_remote(map_to_rank(xs.free_bar, s));
  }
  return mine_row;
}

// One layer of a launch.  The tensor maps live in the kernel parameters.
struct LayerDesc {
  CUtensorMap mg, mp, ma;  // G [B][T][p], P [p][k], A [B][T][d]
  int d, p, nchunks;       // nchunks = projection blocks per sample
  int ready_target;        // ready[l][i] value meaning "W_l,i complete"
  Phase ph1, ph2;
};

template <int CAP>
struct HParams {
  CUtensorMap mw[3];       // the sketch buffers, [B][2k][T_pad] (layer l: l % 3)
  int L, B, T, mtiles;     // layers; batch; tokens; sketch blocks per sample
  int cl;                  // cluster size of the launch
  int maxch;               // stride of chunk_norms per (layer, sample)
  long long tpad;
  __nv_bfloat16* W[3];
  int* ready;              // [L][B]
  int* tickets;            // [L][B]
  int* lticket;            // [B]   layers finished per sample
  int* done2;              // [L]   projection blocks finished per layer
  int* exit_count;         // [1]
  float* chunk_norms;      // [L][B][maxch]
  float* nl;               // [L][B]
  float* n_out;
  int accumulate;
  float norm_scale;                // 1, or 1/k for the +-1 projection
  float clip_C;                    // clip epilogue (c_out non-null): c = min(1, C / sqrt(n))
  float* c_out;
  int32_t* nonfinite;
  unsigned long long seed, step;   // +-1 projection: its Philox stream
  unsigned long long wait_ns;      // limit of every wait in the launch
  // The first two passes of Hutch++ (CAP == kHppCap, see hpp_launch): layer 0
  // is pass 1 (sketch G [S | P], projection A^T W written as Z hi/lo and X P),
  // layer 1 pass 2 (sketch A Z_i, Z_i per sample and summed from its hi/lo
  // halves; projection G^T W written as M fp32 and hi/lo).
  __nv_bfloat16* hz;       // Z hi/lo [B][d][32]
  float* hyp;              // X P [B][d][16]
  float* hm;               // M [B][p][16]
  __nv_bfloat16* hmh;      // M hi/lo [B][p][32]
  int* zdone;              // [B] pass-1 projection blocks written per sample
  int zdone_target;        // their number per sample
  int mdone_target;        // pass-2 projection blocks per sample
  LayerDesc layer[CAP];     // CAP = 1 for single-layer calls: a small parameter block
};

// CAP of the launch that runs the first two passes of Hutch++ (no
// Hutchinson launch has two layer slots: those have 1 or kMaxFusedLayers).
constexpr int kHppCap = 2;

// A tile of a streamed operand (G in a sketch phase, A in a projection phase).
// A Hutchinson launch reads each once, so its lines carry the evict-first L2
// policy and the sketch written between the phases, and P, keep their place
// in L2.  The Hutch++ launch does the same in its sketch phases, but its
// projections leave their operand at the default: the next pass starts by
// reading that operand again (pass 2's sketch the A of pass 1's projection,
// pass 3's sketch the G of pass 2's) and finds its most recent part in L2.
template <int CAP>
__device__ __forceinline__ void load_streamed(void* dst, const CUtensorMap* map, uint64_t* bar,
                                              int c0, int c1, int c2, uint64_t pol, bool sketch) {
  if (CAP == kHppCap && !sketch)
    tma_load_3d(dst, map, bar, c0, c1, c2);
  else
    tma_load_3d_hint(dst, map, bar, c0, c1, c2, pol);
}

// The +-1 projection (reading of papernotes.org, "Experiments > Ablation": a
// {-1, +1} one-bit P instead of a Gaussian one): rows [128 u, 128 u + 128) of
// S [p][K] written by one warp as bf16 +-1 into the P tile of a sketch stage,
// in the layout the TMA gives that tile: MN-major, 2K-byte rows, 64-byte
// swizzle for K = 32 (16-byte chunk c of row r lands at chunk c ^ ((r>>1)&3)),
// 32-byte for K = 16 (chunk c ^ ((r>>2)&1)).  Entry (R, v) is bit (e & 31) of
// word (e >> 5) & 3 of Philox block e >> 7, e = R K + v; bit 1 gives -1.
// part: which of the two writer warps calls (each writes half of every row's
// 16-byte chunks; both compute the same Philox blocks).
template <int K>
__device__ __forceinline__ void gen_sign_tile(uint8_t* tile, int u, int lane, int part,
                                              const RoundKeys& rk, uint64_t step) {
  auto pack = [](uint32_t bits8, int m) {  // two bf16 signs from bits 2m, 2m+1
    const uint32_t b0 = (bits8 >> (2 * m)) & 1u, b1 = (bits8 >> (2 * m + 1)) & 1u;
    return (0x3F80u | (b0 << 15)) | ((0x3F80u | (b1 << 15)) << 16);
  };
  if constexpr (K == 32) {
    // lane l: block 32 u + l = rows 4 l .. 4 l + 3, one word per row
    const uint4 w = philox_block(static_cast<uint64_t>(u) * 32 + lane, step, rk);
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int r = 4 * lane + q;
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = 2 * part + cc;
        const uint32_t b8 = (words[q] >> (8 * c)) & 0xFFu;
        const int pc = c ^ ((r >> 1) & 3);
        *reinterpret_cast<uint4*>(tile + r * 64 + pc * 16) =
            make_uint4(pack(b8, 0), pack(b8, 1), pack(b8, 2), pack(b8, 3));
      }
    }
  } else {
    // lanes 0..15: block 16 u + l = rows 8 l .. 8 l + 7, two rows per word
    if (lane < 16) {
      const uint4 w = philox_block(static_cast<uint64_t>(u) * 16 + lane, step, rk);
      const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int r = 8 * lane + 2 * q + h;
          {
            const int c = part;
            const uint32_t b8 = (words[q] >> (16 * h + 8 * c)) & 0xFFu;
            const int pc = c ^ ((r >> 2) & 1);
            *reinterpret_cast<uint4*>(tile + r * 32 + pc * 16) =
                make_uint4(pack(b8, 0), pack(b8, 1), pack(b8, 2), pack(b8, 3));
          }
        }
      }
    }
  }
}

// Threads per CTA: TMA producer, MMA issuer, four epilogue warps, and with the
// +-1 projection two more warps that write the sign tiles.
template <bool PM1>
constexpr int hutch_threads() { return PM1 ? 256 : 192; }

// Step ps (0 <= ps < 2L) of the one order in which every role of every CTA
// walks the phases of a launch: the sketch of layer 0, then the sketch of
// layer l + 1 before the projection of layer l, and the last projection at
// the end,
//   S0, S1, P0, S2, P1, ..., S(L-1), P(L-2), P(L-1).
// A CTA reaches the projection of layer l one sketch after its own sketch
// blocks of l, so the other CTAs' blocks of l are normally done by then and
// the projection seldom waits.  Every wait is still on a phase that comes
// earlier in this order on every CTA: P(l) on S(l), and S(l), which writes
// sketch buffer l % 3, on P(l - 3), the buffer's previous reader.
template <int CAP>
__device__ __forceinline__ void phase_at(int ps, int L, int& l, bool& sketch) {
  if (CAP == 1) {  // one layer: S0, P0
    l = 0;
    sketch = ps == 0;
  } else if (CAP == kHppCap) {
    // Hutch++ passes 1 and 2: the sketch of pass 2 reads pass 1's projection,
    // so the phases go in order, S0, P0, S1, P1
    l = ps >> 1;
    sketch = (ps & 1) == 0;
  } else if (ps == 0) {
    l = 0;
    sketch = true;
  } else if (ps == 2 * L - 1) {
    l = L - 1;
    sketch = false;
  } else if (ps & 1) {
    l = (ps + 1) >> 1;
    sketch = true;
  } else {
    l = (ps >> 1) - 1;
    sketch = false;
  }
}

template <int K, int CAP, bool PM1>
__global__ void __launch_bounds__(hutch_threads<PM1>(), 1)
    tc_hutch_kernel(const __grid_constant__ HParams<CAP> a) {
  static_assert(!PM1 || CAP == 1, "the +-1 projection runs one layer per launch");
  using Cfg = HCfg<K>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_red[4];

  // The schedule (block split, exchange partners, ready targets) is planned
  // for clusters of a.cl CTAs.  A launch of any other cluster shape would make
  // the exchange address ranks that do not exist: do nothing and say so.
  if (cluster_nctarank() != static_cast<uint32_t>(a.cl)) {
    if (threadIdx.x == 0) record_error(DPRC_DEVERR_LAUNCH);
    return;
  }

  uint8_t* ring = align_1024(smem_raw);
  uint64_t* bars = reinterpret_cast<uint64_t*>(ring + Cfg::kRing);
  uint64_t* full = bars;                  // [kStages]
  uint64_t* empty = full + kStages;       // [kStages]
  uint64_t* accf_r = empty + kStages;     // [2]
  uint64_t* acce_r = accf_r + 2;          // [2]
  uint64_t* accf_c = acce_r + 2;          // [2]
  uint64_t* acce_c = accf_c + 2;          // [2]
  uint64_t* drain = acce_c + 2;           // MMA thread: all its MMAs complete
  Xchg xs;
  xs.recv_bar = acce_c + 3;
  xs.free_bar = acce_c + 4;
  xs.norm_bar = acce_c + 5;  // [2]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cfg::kBars);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  xs.norms = reinterpret_cast<float*>(bars + Cfg::kBars + 2);  // [2][8]
  xs.recv = reinterpret_cast<float*>(ring + Cfg::kRing + Cfg::kCtrl);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a dependent launch (the clip factors, or the next call) may start now;
  // it waits for this grid's completion before touching memory
  pdl_launch_dependents();
  const int nlayers = CAP == 1 ? 1 : a.L;  // a constant for single-layer launches
  const int cl = a.cl;
  const int rank = cl > 1 ? static_cast<int>(cluster_ctarank()) : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // with the +-1 projection a stage also waits for the two sign-tile halves
      mbar_init(&full[s], PM1 ? 3 : 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&accf_r[s], 1);
      mbar_init(&acce_r[s], 4);
      mbar_init(&accf_c[s], 1);
      mbar_init(&acce_c[s], 4);
      mbar_init(&xs.norm_bar[s], cl > 1 ? cl - 1 : 1);
    }
    mbar_init(drain, 1);
    if (cl > 1) {
      mbar_init(xs.recv_bar, (cl - 1) * (kRows / cl));
      mbar_init(xs.free_bar, cl - 1);
    }
    fence_mbar_init();
    *abort_flag = 0;
  }
  // The producer (thread 0, which initialised the barriers) issues the first
  // ring slots of its first sketch block before the CTA barrier, so their
  // DRAM round trip overlaps the TMEM allocation and the barrier.  Launched as
  // a programmatic dependent of the previous kernel in the stream, this grid
  // may start while that one finishes: thread 0 first waits until it has
  // completed and its writes are visible (every other thread touches memory
  // only after the CTA barrier below, behind this wait); the barrier set-up
  // above and the TMEM allocation overlap the previous grid's tail.
  int pre = 0;
  if (threadIdx.x == 0) pdl_wait();
  if (threadIdx.x == 0) {
    const LayerDesc& L0 = a.layer[0];
    const Mine m1 = mine(L0.ph1, cl, rank);
    const uint64_t pol = l2_policy_evict_first();
    if (count_blocks(L0.ph1, m1) > 0) {
      const long long b = m1.first;
      const int i = static_cast<int>(b / a.mtiles);
      const int t0 = static_cast<int>(b - static_cast<long long>(i) * a.mtiles) * kTok;
      for (int u = m1.ulo; u < m1.uhi && pre < kStages; ++u, ++pre) {
        uint8_t* slot = ring + pre * Cfg::kSlot;
        mbar_arrive_expect_tx(&full[pre], PM1 ? Cfg::kRowG : Cfg::kRowStage);
#pragma unroll
        for (int h = 0; h < 2; ++h)
          load_streamed<CAP>(slot + h * Cfg::kRowGBox, &L0.mg, &full[pre],
                             rot_unit(m1, u) * kCol + h * 64, t0, i, pol, true);
        if (!PM1) tma_load_3d(slot + Cfg::kRowG, &L0.mp, &full[pre], 0, rot_unit(m1, u) * kCol, 0);
      }
    }
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&a.mw[0]);
    if (CAP > 1) {
      tma_prefetch_desc(&a.mw[1]);
      tma_prefetch_desc(&a.mw[2]);
    }
    for (int l = 0; l < nlayers && l < 4; ++l) {
      const LayerDesc& Ld = a.layer[CAP == 1 ? 0 : l];
      tma_prefetch_desc(&Ld.mg);
      if (!PM1) tma_prefetch_desc(&Ld.mp);
      tma_prefetch_desc(&Ld.ma);
    }
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
  // The waits on other CTAs' progress (sketch ready, sketch buffer free) end
  // within a.wait_ns; every wait inside the CTA or its cluster within twice
  // that.  Those are downstream of the former (a tile waits for the sketch
  // its W half needs, a peer's partials for the peer's tiles) and may start
  // earlier, so the longer limit lets the wait that is the cause run out
  // first and record its code.  The pipeline waits also end as soon as
  // another role has set abort_flag, so after the first failure the roles
  // unwind without each running out its own limit; the exchange waits do not
  // (both ranks of a cluster always run the same exchanges).
  const unsigned long long lim = a.wait_ns;
  const unsigned long long lim2 = 2 * a.wait_ns;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      bool ok = true;
      long long it = 0;  // stages issued (both phases, all layers)
      const uint64_t pol = l2_policy_evict_first();
      auto take_slot = [&](long long i) -> int {
        const int s = static_cast<int>(i % kStages);
        if (!mbar_wait_lim(&empty[s], (static_cast<uint32_t>(i / kStages) & 1) ^ 1,
                           DPRC_DEVERR_PIPE_EMPTY, lim2, abort_flag))
          ok = false;
        return s;
      };
      #pragma unroll(CAP == 1 ? 2 : 1)
      for (int ps = 0; ps < 2 * nlayers && ok; ++ps) {
        int l;
        bool sketch;
        phase_at<CAP>(ps, nlayers, l, sketch);
        const LayerDesc& Ld = a.layer[CAP == 1 ? 0 : l];
        if (sketch) {
          if (CAP > 1 && l + 4 < nlayers) {
            const LayerDesc& Ln = a.layer[CAP == 1 ? 0 : l + 4];
            tma_prefetch_desc(&Ln.mg);
            tma_prefetch_desc(&Ln.mp);
            tma_prefetch_desc(&Ln.ma);
          }
          // phase 1: G and P tiles
          const Mine m1 = mine(Ld.ph1, cl, rank);
          const long long nb1 = count_blocks(Ld.ph1, m1);
          // Hutch++ pass 2: the operand Z_i is per sample (its batch coordinate)
          // and written by pass 1's projection, waited for per sample
          const bool zbatched = CAP == kHppCap && l == 1;
          int z_i = -1;
          for (long long j = 0; j < nb1 && ok; ++j) {
            const long long b = m1.first + j * m1.step;
            const int i = static_cast<int>(b / a.mtiles);
            const int t0 = static_cast<int>(b - static_cast<long long>(i) * a.mtiles) * kTok;
            if (zbatched && i != z_i) {
              if (DPRC_IN(i >= 0 && i < a.B) &&
                  wait_geq(&a.zdone[i], a.zdone_target, lim, abort_flag)) {
                fence_proxy_async_global();
              } else {
                ok = false;
                break;
              }
              z_i = i;
            }
            for (int u = m1.ulo; u < m1.uhi; ++u) {
              if (it < pre) {  // issued before the CTA barrier
                ++it;
                continue;
              }
              const int s = take_slot(it);
              if (!ok) break;
              uint8_t* slot = ring + s * Cfg::kSlot;
              // (+-1 projection: the sign tile comes from the generator warp)
              mbar_arrive_expect_tx(&full[s], PM1 ? Cfg::kRowG : Cfg::kRowStage);
  #pragma unroll
              for (int h = 0; h < 2; ++h)
                load_streamed<CAP>(slot + h * Cfg::kRowGBox, &Ld.mg, &full[s],
                                   rot_unit(m1, u) * kCol + h * 64, t0, i, pol, true);
              if (!PM1)
                tma_load_3d(slot + Cfg::kRowG, &Ld.mp, &full[s], 0, rot_unit(m1, u) * kCol,
                            zbatched ? i : 0);
              ++it;
            }
          }
        } else {
          // phase 2: A tiles, then, once sample i's sketch is complete, W tiles.
          // Before waiting for a new sample's sketch, up to kStages stages of A
          // go out; otherwise the A and W tiles of a stage go out together.  Two
          // cursors walk the stages (one division per block: this thread paces
          // the whole pipeline).
          const Mine m2 = mine(Ld.ph2, cl, rank);
          const long long nb2 = count_blocks(Ld.ph2, m2);
          const int nu2 = m2.uhi - m2.ulo;
          const long long total2 = nb2 * nu2;
          struct Cursor {
            long long j = 0;
            int u = 0, i = 0, ch = 0;
          };
          auto seek = [&](Cursor& c) {
            const long long b = m2.first + c.j * m2.step;
            c.i = static_cast<int>(b / Ld.nchunks);
            c.ch = static_cast<int>(b - static_cast<long long>(c.i) * Ld.nchunks);
          };
          auto advance = [&](Cursor& c) {
            if (++c.u == m2.uhi) {
              c.u = m2.ulo;
              ++c.j;
              if (c.j < nb2) seek(c);
            }
          };
          Cursor ca, cw;
          ca.u = cw.u = m2.ulo;
          if (nb2 > 0) {
            seek(ca);
            seek(cw);
          }
          const long long base = it;     // global index of this phase's first stage
          long long w_done = 0;          // stages of this phase with W issued
          int ready_i = -1;
          while (w_done < total2) {
            const bool need_wait = ok && cw.i != ready_i;
            const long long ahead = need_wait ? kStages : 1;
            const long long a_to = w_done + ahead < total2 ? w_done + ahead : total2;
            while (ok && it - base < a_to) {
              const int s = take_slot(it);
              if (!ok) break;
              uint8_t* slot = ring + s * Cfg::kSlot;
              mbar_arrive_expect_tx(&full[s], Cfg::kColStage);
              if (PM1) {  // no sign tile in a projection stage
                mbar_arrive(&full[s]);
                mbar_arrive(&full[s]);
              }
  #pragma unroll
              for (int h = 0; h < 2; ++h)
                load_streamed<CAP>(slot + h * Cfg::kColABox, &Ld.ma, &full[s], ca.ch * kRows + h * 64,
                                   ca.u * kTok, ca.i, pol, false);
              ++it;
              advance(ca);
            }
            if (w_done >= it - base) break;  // nothing left to complete (after an error)
            if (need_wait && !DPRC_IN(cw.i >= 0 && cw.i < a.B && l < a.L)) ok = false;
            if (need_wait && ok) {
              if (wait_geq(&a.ready[l * a.B + cw.i], Ld.ready_target, lim, abort_flag)) {
                fence_proxy_async_global();
                ready_i = cw.i;
              } else {
                ok = false;  // still load W so the issued stages complete; results are void
              }
            }
            const long long g = base + w_done;
            const int s = static_cast<int>(g % kStages);
            uint8_t* slot = ring + s * Cfg::kSlot;
  #pragma unroll
            for (int h = 0; h < 2; ++h)
              tma_load_3d(slot + Cfg::kColA + h * Cfg::kColWBox, &a.mw[l % 3], &full[s],
                          cw.u * kTok + h * 64, 0, cw.i);
            ++w_done;
            advance(cw);
          }
        }
      }
      if (!ok) *abort_flag = 1;
      // Let every copy this thread issued land before the CTA can exit.  Only
      // the last kStages stages can be in flight: each earlier one was
      // consumed (its slot was freed) before its slot was refilled.
      for (long long k = it - 1; k >= 0 && k >= it - kStages; --k)
        mbar_wait_lim(&full[k % kStages], static_cast<uint32_t>(k / kStages) & 1,
                      DPRC_DEVERR_PIPE_FULL, lim2, nullptr);
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      bool ok = true;
      bool issued = false;  // any MMA issued (to drain before the CTA exits)
      long long it = 0, seg1 = 0, seg2 = 0;
      constexpr uint32_t idesc1 = make_idesc_bf16(128, Cfg::kNR, false, true);
      constexpr uint32_t p_swz = swz_code_for_bytes(2 * Cfg::kNR);
      constexpr uint32_t idesc2 = make_idesc_bf16(128, Cfg::kNC, true, false);
      auto wait_full = [&](long long i) -> int {
        const int s = static_cast<int>(i % kStages);
        if (!mbar_wait_lim(&full[s], static_cast<uint32_t>(i / kStages) & 1,
                           DPRC_DEVERR_PIPE_FULL, lim2, abort_flag))
          ok = false;
        return s;
      };
      #pragma unroll(CAP == 1 ? 2 : 1)
      for (int ps = 0; ps < 2 * nlayers && ok; ++ps) {
        int l;
        bool sketch;
        phase_at<CAP>(ps, nlayers, l, sketch);
        const LayerDesc& Ld = a.layer[CAP == 1 ? 0 : l];
        if (sketch) {
          const Mine m1 = mine(Ld.ph1, cl, rank);
          const long long nb1 = count_blocks(Ld.ph1, m1);
          for (long long j = 0; j < nb1 && ok; ++j, ++seg1) {
            const int abuf = static_cast<int>(seg1 & 1);
            if (!mbar_wait_lim(&acce_r[abuf], (static_cast<uint32_t>(seg1 >> 1) & 1) ^ 1,
                               DPRC_DEVERR_ACCUM, lim2, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int u = m1.ulo; u < m1.uhi; ++u, ++it) {
              const int s = wait_full(it);
              if (!ok) break;
              tc_fence_after();
              const uint32_t ga = smem_u32(ring + s * Cfg::kSlot);
              const uint32_t pa = ga + Cfg::kRowG;
  #pragma unroll
              for (int kk = 0; kk < kCol / 16; ++kk) {
                // G: two boxes of 128 token rows x 64 p, K-major, 128-byte swizzle.
                const uint64_t ad =
                    make_sdesc(ga + (kk >> 2) * Cfg::kRowGBox + (kk & 3) * 32, 16, 1024, kSwz128);
                // P: 128 p rows x K columns, MN-major, one swizzle atom wide.
                const uint64_t bd = make_sdesc(pa + kk * 32 * Cfg::kNR, 16, 16 * Cfg::kNR, p_swz);
                umma_bf16(tmem + abuf * Cfg::kAccR, ad, bd, idesc1,
                          (u == m1.ulo && kk == 0) ? 0u : 1u);
              }
              issued = true;
              umma_commit(&empty[s]);
            }
            if (ok) umma_commit(&accf_r[abuf]);
          }
        } else {
          const Mine m2 = mine(Ld.ph2, cl, rank);
          const long long nb2 = count_blocks(Ld.ph2, m2);
          for (long long j = 0; j < nb2 && ok; ++j, ++seg2) {
            const int abuf = static_cast<int>(seg2 & 1);
            if (!mbar_wait_lim(&acce_c[abuf], (static_cast<uint32_t>(seg2 >> 1) & 1) ^ 1,
                               DPRC_DEVERR_ACCUM, lim2, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            for (int u = m2.ulo; u < m2.uhi; ++u, ++it) {
              const int s = wait_full(it);
              if (!ok) break;
              tc_fence_after();
              const uint32_t xa = smem_u32(ring + s * Cfg::kSlot);
              const uint32_t wa = xa + Cfg::kColA;
  #pragma unroll
              for (int kk = 0; kk < kTok / 16; ++kk) {
                // A^T: 128 d (two 64-d atoms, LBO = one box) x 16 tokens (SBO 1 KB).
                const uint64_t ad = make_sdesc(xa + kk * 2048, Cfg::kColABox, 1024, kSwz128);
                // Sketch: 2K rows x 64 tokens per box, K-major, 128-byte swizzle.
                const uint64_t bd =
                    make_sdesc(wa + (kk >> 2) * Cfg::kColWBox + (kk & 3) * 32, 16, 1024, kSwz128);
                umma_bf16(tmem + Cfg::kColAcc0 + abuf * Cfg::kNC, ad, bd, idesc2,
                          (u == m2.ulo && kk == 0) ? 0u : 1u);
              }
              issued = true;
              umma_commit(&empty[s]);
            }
            if (ok) umma_commit(&accf_c[abuf]);
          }
        }
      }
      if (!ok) *abort_flag = 1;
      // On every path (a wait that gave up skips the accumulator commits): no
      // MMA may still write tensor memory once the CTA releases it.
      if (issued) umma_drain(drain, lim2);
    }
  } else if (PM1 && warp >= 6) {
    // ---------------- sign-tile writers (+-1 projection, one layer) ----------------
    // Walks the sketch stages in the producer's order; once a slot is free it
    // writes that stage's signs, makes them visible to the tensor cores (async
    // proxy) and gives the stage's second arrival.
    const RoundKeys rk = round_keys(a.seed);
    const LayerDesc& Ld = a.layer[0];
    const Mine m1 = mine(Ld.ph1, cl, rank);
    const long long nb1 = count_blocks(Ld.ph1, m1);
    long long it = 0;
    bool ok = true;
    for (long long j = 0; j < nb1 && ok; ++j) {
      for (int u = m1.ulo; u < m1.uhi; ++u, ++it) {
        const int s = static_cast<int>(it % kStages);
        bool free_ok = true;
        if (lane == 0)
          free_ok = mbar_wait_lim(&empty[s], (static_cast<uint32_t>(it / kStages) & 1) ^ 1,
                                  DPRC_DEVERR_PIPE_EMPTY, lim2, abort_flag);
        ok = __shfl_sync(0xffffffffu, free_ok ? 1 : 0, 0) != 0 && *abort_flag == 0;
        if (!ok) break;
        gen_sign_tile<K>(ring + s * Cfg::kSlot + Cfg::kRowG, rot_unit(m1, u), lane, warp - 6, rk,
                         a.step);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&full[s]);
      }
    }
  } else if (warp < 6) {
    // ---------------- epilogue warps 2..5 ----------------
    const int ew = warp - 2;
    const int q = warp & 3;         // TMEM lane quadrant of this warp
    const int row = q * 32 + lane;  // row of the 128-row tile = TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    bool ok = true;
    long long seg1 = 0, seg2 = 0;
    // split projection blocks so far: the same sequence on every rank of the
    // cluster (seg2 also counts whole blocks, whose number differs by CTA)
    long long nsplit2 = 0;
    int rnd = 0;  // cluster exchange rounds so far
    int rounds = 0;
    for (int l = 0; l < nlayers; ++l) {
      const LayerDesc& Ld = a.layer[CAP == 1 ? 0 : l];
      if (Ld.ph1.split) rounds += static_cast<int>(count_blocks(Ld.ph1, mine(Ld.ph1, cl, rank)));
      if (Ld.ph2.split) rounds += static_cast<int>(count_blocks(Ld.ph2, mine(Ld.ph2, cl, rank)));
    }
    #pragma unroll(CAP == 1 ? 2 : 1)
    for (int ps = 0; ps < 2 * nlayers; ++ps) {
      int l;
      bool sketch;
      phase_at<CAP>(ps, nlayers, l, sketch);
      const LayerDesc& Ld = a.layer[CAP == 1 ? 0 : l];
      if (sketch) {
        __nv_bfloat16* W = a.W[l % 3];
        // phase 1: sketch rows -> W hi/lo, then count the block done
        const Mine m1 = mine(Ld.ph1, cl, rank);
        const long long nb1 = count_blocks(Ld.ph1, m1);
        if (CAP > 1 && nb1 > 0 && l >= 3) {
          // the previous user of this sketch buffer (layer l - 3) must be done
          if (threadIdx.x == 64 && ok &&
              (!DPRC_IN(l < a.L) ||
               !wait_geq(&a.done2[l - 3],
                         static_cast<int>(a.layer[CAP == 1 ? 0 : l - 3].ph2.nblocks), lim,
                         abort_flag)))
            *abort_flag = 1;
          named_bar_sync(1, 128);
        }
        for (long long j = 0; j < nb1; ++j, ++seg1) {
          const int abuf = static_cast<int>(seg1 & 1);
          bool live = ok &&
                      mbar_wait_lim(&accf_r[abuf], static_cast<uint32_t>(seg1 >> 1) & 1,
                                    DPRC_DEVERR_ACCUM, lim2, abort_flag) &&
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
          if (Ld.ph1.split) {
            mine_row = xchg_rows<K>(xs, cl, rank, row, rnd, rnd + 1 == rounds, y, ok, lim2);
            ++rnd;
          }
          if (CAP == kHppCap && l == 1) {
            // Hutch++ pass 2: the operand's columns are Z_hi | Z_lo, so the
            // sketch is the sum of the two halves; the other half stays zero
            // (rows K/2..K-1 of each plane of W, which the projection's MMA
            // reads as zero columns)
  #pragma unroll
            for (int c = 0; c < K / 2; ++c) {
              y[c] += y[K / 2 + c];
              y[K / 2 + c] = 0.f;
            }
          }
          const long long b = m1.first + j * m1.step;
          const int i = static_cast<int>(b / a.mtiles);
          const int t = static_cast<int>(b - static_cast<long long>(i) * a.mtiles) * kTok + row;
          if (mine_row && ok && t < a.T && DPRC_IN(i >= 0 && i < a.B && t < a.tpad)) {
            __nv_bfloat16* wi = W + static_cast<size_t>(i) * 2 * K * a.tpad + t;
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
          if (ew == 0 && lane == 0 && ok && DPRC_IN(i >= 0 && i < a.B && l < a.L)) {
            __threadfence();
            atomicAdd(&a.ready[l * a.B + i], 1);
          }
        }
      } else {
        // phase 2: squared norms of the projection blocks
        const Mine m2 = mine(Ld.ph2, cl, rank);
        const long long nb2 = count_blocks(Ld.ph2, m2);
        for (long long j = 0; j < nb2; ++j, ++seg2) {
          const int abuf = static_cast<int>(seg2 & 1);
          bool live = ok &&
                      mbar_wait_lim(&accf_c[abuf], static_cast<uint32_t>(seg2 >> 1) & 1,
                                    DPRC_DEVERR_ACCUM, lim2, abort_flag) &&
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
          if (Ld.ph2.split) {
            mine_row = xchg_rows<K>(xs, cl, rank, row, rnd, rnd + 1 == rounds, y, ok, lim2);
            ++rnd;
          }
          const long long b = m2.first + j * m2.step;
          const int i = static_cast<int>(b / Ld.nchunks);
          const int ch = static_cast<int>(b - static_cast<long long>(i) * Ld.nchunks);
          if constexpr (CAP == kHppCap) {
            // Hutch++ passes 1 and 2: this rank's rows of the projection go to
            // memory (pass 1: Z = columns 0..15 as hi/lo, X P = 16..31 in
            // fp32; pass 2: M in fp32 and hi/lo), then one count per block
            constexpr int H = K / 2;
            const int grow = ch * kRows + row;
            if (mine_row && ok && grow < Ld.d && DPRC_IN(i >= 0 && i < a.B)) {
              const size_t yrow = static_cast<size_t>(i) * Ld.d + grow;
              float yh[H];
  #pragma unroll
              for (int c = 0; c < H; ++c) yh[c] = y[c];
              float4* f4 = reinterpret_cast<float4*>((l == 0 ? a.hyp : a.hm) + yrow * H);
  #pragma unroll
              for (int c4 = 0; c4 < H / 4; ++c4) {
                const int c = (l == 0 ? H : 0) + 4 * c4;
                f4[c4] = make_float4(y[c], y[c + 1], y[c + 2], y[c + 3]);
              }
              store_hilo_row<H>((l == 0 ? a.hz : a.hmh) + yrow * K, yh);
            }
            fence_proxy_async_global();  // Z is read by TMA in pass 2's sketch
            named_bar_sync(1, 128);
            if (threadIdx.x == 64 && ok && DPRC_IN(i >= 0 && i < a.B)) {
              __threadfence();
              if (l == 0) {
                // the sample's last pass-1 block: every block of the sample has
                // passed its wait on ready[0][i]
                if (atomicAdd(&a.zdone[i], 1) == a.zdone_target - 1) a.ready[i] = 0;
              } else if (atomicAdd(&a.tickets[a.B + i], 1) == a.mdone_target - 1) {
                // the sample's last pass-2 block: every block of pass 2 has
                // passed its waits, on zdone[i] (sketch) and ready[1][i]
                a.tickets[a.B + i] = 0;
                a.ready[a.B + i] = 0;
                a.zdone[i] = 0;
              }
            }
            named_bar_sync(1, 128);
            continue;
          }
          float sq = 0.f;
          if (mine_row && ok && ch * kRows + row < Ld.d) {
  #pragma unroll
            for (int t = 0; t < K; ++t) sq = fmaf(y[t], y[t], sq);
            sq *= a.norm_scale;  // 1, or 1/k (a power of two: exact)
          }
  #pragma unroll
          for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
          if (lane == 0) s_red[ew] = sq;
          named_bar_sync(1, 128);
          if (ew == 0) {
            // warp 2: lane 0 gathers the block's norm; the whole warp finishes
            // a sample (the chunk and layer sums read many L2 lines: one per lane)
            const float part = (s_red[0] + s_red[1]) + (s_red[2] + s_red[3]);
            float chunk = part;
            int leader = 1;
            if (lane == 0 && Ld.ph2.split) {
              float* nb = xs.norms + (nsplit2 & 1) * 8;
              if (rank != 0) {
                if (DPRC_IN(rank < 8)) {
                  st_cluster_f32(map_to_rank(nb + rank, 0), part);
                  mbar_arrive_remote(map_to_rank(&xs.norm_bar[nsplit2 & 1], 0));
                }
                leader = 0;
              } else {
                if (!mbar_wait_cluster(&xs.norm_bar[nsplit2 & 1],
                                       static_cast<uint32_t>(nsplit2 >> 1) & 1, DPRC_DEVERR_CLUSTER,
                                       lim2))
                  ok = false;
                nb[0] = part;
                chunk = 0.f;
                for (int s = 0; s < cl; ++s) chunk += nb[s];
              }
            }
            leader = __shfl_sync(0xffffffffu, leader, 0);
            const bool lok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!lok) ok = false;
            if (leader && lok &&
                DPRC_IN(i >= 0 && i < a.B && ch >= 0 && ch < Ld.nchunks && Ld.nchunks <= a.maxch)) {
              const size_t li = static_cast<size_t>(l) * a.B + i;
              int last = 0;
              if (lane == 0) {
                a.chunk_norms[li * a.maxch + ch] = chunk;
                __threadfence();
                last = atomicAdd(&a.tickets[li], 1) == Ld.nchunks - 1;
              }
              if (__shfl_sync(0xffffffffu, last, 0)) {
                // last block of (layer l, sample i): its norm, summed in a fixed order
                __threadfence();
                float sum = 0.f;
                for (int c = lane; c < Ld.nchunks; c += 32) sum += __ldcg(&a.chunk_norms[li * a.maxch + c]);
  #pragma unroll
                for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
                int final_layer = 0;
                if (lane == 0) {
                  a.tickets[li] = 0;
                  a.ready[li] = 0;
                  if (CAP == 1) {
                    // one layer: no layer sum to wait for
                    const float nv = (a.accumulate ? a.n_out[i] : 0.f) + sum;
                    a.n_out[i] = nv;
                    if (a.c_out != nullptr) {
                      bool bad;
                      a.c_out[i] = clip_factor(nv, a.clip_C, bad);
                      if (bad && a.nonfinite != nullptr) atomicAdd(a.nonfinite, 1);
                    }
                  } else {
                    a.nl[li] = sum;
                    __threadfence();
                    final_layer = atomicAdd(&a.lticket[i], 1) == a.L - 1;
                  }
                }
                if (CAP > 1 && __shfl_sync(0xffffffffu, final_layer, 0)) {
                  // last layer of sample i: the layer sum, in a fixed order
                  __threadfence();
                  float tot = 0.f;
                  for (int ll = lane; ll < a.L; ll += 32)
                    tot += __ldcg(&a.nl[static_cast<size_t>(ll) * a.B + i]);
  #pragma unroll
                  for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
                  if (lane == 0) {
                    const float nv = (a.accumulate ? a.n_out[i] : 0.f) + tot;
                    a.n_out[i] = nv;
                    a.lticket[i] = 0;
                    if (a.c_out != nullptr) {
                      bool bad;
                      a.c_out[i] = clip_factor(nv, a.clip_C, bad);
                      if (bad && a.nonfinite != nullptr) atomicAdd(a.nonfinite, 1);
                    }
                  }
                }
              }
              // this block no longer reads the sketch buffer of layer l
              if (CAP > 1 && lane == 0 && DPRC_IN(l < a.L)) atomicAdd(&a.done2[l], 1);
            }
          }
          named_bar_sync(1, 128);
          if (Ld.ph2.split) ++nsplit2;
        }
      }
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
  if (CAP > 1 && threadIdx.x == 0) {
    // the last CTA out clears the per-layer projection counts for the next call
    __threadfence();
    if (atomicAdd(a.exit_count, 1) == static_cast<int>(gridDim.x) - 1) {
      for (int l = 0; l < a.L; ++l) a.done2[l] = 0;
      *a.exit_count = 0;
    }
  }
}

template <int K, int CAP, bool PM1>
cudaError_t set_smem_once() {
  constexpr int kMaxDev = 64;
  static std::atomic<int> done[kMaxDev];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < kMaxDev && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(tc_hutch_kernel<K, CAP, PM1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           HCfg<K>::smem(8));
  if (e == cudaSuccess && dev >= 0 && dev < kMaxDev) done[dev].store(1, std::memory_order_release);
  return e;
}

// CTAs of this kernel that may run at once in one launch with clusters of
// cl: the driver's occupancy figures (one CTA per SM), cached per device and
// cl.
template <int K, int CAP, bool PM1>
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
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tc_hutch_kernel<K, CAP, PM1>,
                                                      hutch_threads<PM1>(),
                                                      smem) != cudaSuccess)
      return 0;
    v = per_sm * device_sm_count();
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cl * device_sm_count());
    cfg.blockDim = dim3(hutch_threads<PM1>());
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = cl;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int ncl = 0;
    if (cudaOccupancyMaxActiveClusters(&ncl, tc_hutch_kernel<K, CAP, PM1>, &cfg) != cudaSuccess)
      return 0;
    v = ncl * cl;
  }
  cache[dev][ci].store(v, std::memory_order_release);
  return v;
}

// Launch of a planned schedule.  The grid is at most what fits on the device
// at once (one CTA per SM; with clusters, the clusters the occupancy query of
// resident_ctas counts), so every CTA is resident together, which the
// cross-CTA waits rely on; when other work holds SMs, a waiting CTA's wait
// ends within its limit with DPRC_DEVERR_READY instead of hanging.  Without
// clusters the launch is a programmatic dependent of the previous kernel in
// the stream: its CTAs may start on SMs that kernel has released, set up, and
// wait for its completion (griddepcontrol.wait) before any memory access.
// Every CTA of the previous grid is already resident when this one starts
// (its CTAs allow the dependent launch only once all of them run), so the
// early CTAs cannot keep it from finishing.  With clusters the launch is a
// plain cluster launch.  Cooperative and cluster attributes are never
// combined: that combination is the one launch form of this kernel that
// faulted the GPU (under a profiler's replay).
// `test_cl` > 0 (failure-detection test only): launch with clusters of that
// size whatever the plan says.
template <int K, int CAP, bool PM1>
cudaError_t launch_k(const HParams<CAP>& a, int grid, cudaStream_t s, int test_cl = 0) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(hutch_threads<PM1>());
  cfg.dynamicSmemBytes = HCfg<K>::smem(a.cl);
  cfg.stream = s;
  const int cl = test_cl > 0 ? test_cl : a.cl;
  cudaLaunchAttribute attr[1];
  if (cl > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
  } else {
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
  }
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, tc_hutch_kernel<K, CAP, PM1>, a);
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

// Devices on which the launch was refused once keep using the two-kernel
// path.
constexpr int kMaxDevices = 64;
std::atomic<int> g_refused[kMaxDevices];

// Schedule of one launch over layers [0, L): the phases of every layer, the
// cluster size and the grid.  False when the kernel cannot run here.
template <int CAP, bool PM1>
bool plan_fused(int L, const int64_t* d, const int64_t* p, int64_t B, int64_t T, int64_t k,
                HParams<CAP>& a, int& grid_out) {
  if (!fused_hutch_supported(k) || L < 1 || L > CAP) return false;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
  if (g_refused[dev].load(std::memory_order_acquire)) return false;
  const int ik = static_cast<int>(k);
  const int slots = device_sm_count();  // one CTA per SM
  a.L = L;
  a.B = static_cast<int>(B);
  a.T = static_cast<int>(T);
  a.mtiles = static_cast<int>((T + kTok - 1) / kTok);
  int cl = 1, maxch = 1;
  for (int l = 0; l < L; ++l) {
    LayerDesc& Ld = a.layer[l];
    Ld.d = static_cast<int>(d[l]);
    Ld.p = static_cast<int>(p[l]);
    Ld.nchunks = static_cast<int>((d[l] + kRows - 1) / kRows);
    Ld.ph1.nblocks = B * a.mtiles;
    Ld.ph1.upb = static_cast<int>((p[l] + kCol - 1) / kCol);
    Ld.ph2.nblocks = B * Ld.nchunks;
    Ld.ph2.upb = a.mtiles;
    const int c1 = want_cl(Ld.ph1.nblocks, Ld.ph1.upb, slots);
    const int c2 = want_cl(Ld.ph2.nblocks, Ld.ph2.upb, slots);
    Ld.ph1.split = c1;  // the wanted cluster size, until cl is known
    Ld.ph2.split = c2;
    cl = c1 > cl ? c1 : cl;
    cl = c2 > cl ? c2 : cl;
    maxch = Ld.nchunks > maxch ? Ld.nchunks : maxch;
  }
  if ((ik == 16 ? set_smem_once<16, CAP, PM1>() : set_smem_once<32, CAP, PM1>()) != cudaSuccess)
    return false;
  const int resident =
      ik == 16 ? resident_ctas<16, CAP, PM1>(cl) : resident_ctas<32, CAP, PM1>(cl);
  if (resident < cl) return false;
  for (int l = 0; l < L; ++l) {
    LayerDesc& Ld = a.layer[l];
    Ld.ph1.split = Ld.ph1.split > 1 && Ld.ph1.upb >= cl ? 1 : 0;
    Ld.ph2.split = Ld.ph2.split > 1 && Ld.ph2.upb >= cl ? 1 : 0;
    Ld.ready_target = a.mtiles * (Ld.ph1.split ? cl : 1);
  }
  // Grid: the multiple of cl (up to what is resident) that minimises the
  // bytes the busiest CTA streams over all phases of all layers (a sketch
  // unit is 32 KB of G, a projection unit 32 KB of A); ties go to the smaller
  // grid.
  long long grid = 0, best = -1;
  for (long long ncl = 1; ncl * cl <= resident; ++ncl) {
    const long long g = ncl * cl;
    auto busiest = [&](const Phase& ph) {
      if (ph.split) return (ph.nblocks + ncl - 1) / ncl * ((ph.upb + cl - 1) / cl);
      return (ph.nblocks + g - 1) / g * ph.upb;
    };
    long long cost = 0;
    for (int l = 0; l < L; ++l) cost += busiest(a.layer[l].ph1) + busiest(a.layer[l].ph2);
    if (best < 0 || cost < best) {
      best = cost;
      grid = g;
    }
  }
  if (grid < cl) return false;
  a.cl = cl;
  a.maxch = maxch;
  grid_out = static_cast<int>(grid);
  return true;
}

}  // namespace

cudaError_t read_device_error_hutch(int32_t* out, bool reset) {
  return read_tu_device_error(out, reset);
}

bool fused_hutch_supported(int64_t k) { return k == 16 || k == 32; }

bool fused_hutch_planned(int64_t B, int64_t T, int64_t d, int64_t p, int64_t k) {
  HParams<1> a;
  int grid = 0;
  return plan_fused<1, false>(1, &d, &p, B, T, k, a, grid);
}

namespace {

template <int CAP, bool PM1>
cudaError_t launch_cap(int L, const void* const* A, const void* const* G, const void* const* P,
                       const int64_t* d, const int64_t* p, int64_t B, int64_t T, int64_t k,
                       const FusedScratch& ws, float* n_out, int accumulate, uint64_t seed,
                       uint64_t step, cudaStream_t s, bool* launched,
                       const ClipOut* clip, const HutchFaultTest* test = nullptr) {
  static thread_local HParams<CAP> a;  // up to ~26 KB: kept off the stack
  int grid = 0;
  if (!plan_fused<CAP, PM1>(L, d, p, B, T, k, a, grid)) return cudaSuccess;
  int test_cl = 0;
  a.wait_ns = kWaitLimitNs;
  if (test != nullptr) {
    a.wait_ns = test->wait_ns;
    if (test->mode == kFaultReadyNeverMet) {
      for (int l = 0; l < L; ++l) a.layer[l].ready_target += 1;  // one more than phase 1 adds
    } else {
      if (a.cl != 1) return cudaSuccess;  // needs a plan without clusters
      test_cl = 2;
      grid += grid & 1;  // a whole number of clusters
    }
  }
  const int ik = static_cast<int>(k);
  a.tpad = ws.tpad;
  for (int b = 0; b < 3; ++b) a.W[b] = static_cast<__nv_bfloat16*>(ws.W[b]);
  a.ready = ws.ready;
  a.tickets = ws.tickets;
  a.lticket = ws.lticket;
  a.done2 = ws.done2;
  a.exit_count = ws.exit_count;
  a.chunk_norms = ws.chunk_norms;
  a.nl = ws.nl;
  a.n_out = n_out;
  a.accumulate = accumulate;
  a.norm_scale = PM1 ? 1.0f / static_cast<float>(k) : 1.0f;
  a.clip_C = clip != nullptr ? clip->C : 0.f;
  a.c_out = clip != nullptr ? clip->c : nullptr;
  a.nonfinite = clip != nullptr ? clip->nonfinite : nullptr;
  a.seed = seed;
  a.step = step;
  for (int b = 0; b < 3; ++b)
    if (!make_tmap_3d_bf16(&a.mw[b], ws.W[b], T, 2 * ik, B, ws.tpad, 2 * ik * ws.tpad, 64,
                           2 * ik, 128))
      return cudaErrorInvalidValue;
  for (int l = 0; l < L; ++l) {
    LayerDesc& Ld = a.layer[l];
    if (!make_tmap_3d_bf16(&Ld.mg, G[l], p[l], T, B, p[l], T * p[l], 64, kTok, 128) ||
        (!PM1 && !make_tmap_3d_bf16(&Ld.mp, P[l], ik, p[l], 1, ik, p[l] * ik, ik, kCol, 2 * ik)) ||
        !make_tmap_3d_bf16(&Ld.ma, A[l], d[l], T, B, d[l], T * d[l], 64, kTok, 128))
      return cudaErrorInvalidValue;
  }
  const cudaError_t e = ik == 16 ? launch_k<16, CAP, PM1>(a, grid, s, test_cl)
                                 : launch_k<32, CAP, PM1>(a, grid, s, test_cl);
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

}  // namespace

cudaError_t launch_tc_hutch_layers(int L, const void* const* A, const void* const* G,
                                   const void* const* P, const int64_t* d, const int64_t* p,
                                   int64_t B, int64_t T, int64_t k, const FusedScratch& ws,
                                   float* n_out, int accumulate, cudaStream_t s,
                                   bool* launched, const ClipOut* clip) {
  *launched = false;
  if (L == 1)
    return launch_cap<1, false>(L, A, G, P, d, p, B, T, k, ws, n_out, accumulate, 0, 0, s,
                                launched, clip);
  return launch_cap<kMaxFusedLayers, false>(L, A, G, P, d, p, B, T, k, ws, n_out, accumulate, 0,
                                            0, s, launched, clip);
}

cudaError_t launch_tc_hutch_fault_test(int L, const void* const* A, const void* const* G,
                                       const void* const* P, const int64_t* d, const int64_t* p,
                                       int64_t B, int64_t T, int64_t k, const FusedScratch& ws,
                                       float* n_out, const HutchFaultTest& test, cudaStream_t s,
                                       bool* launched) {
  *launched = false;
  if (L == 1)
    return launch_cap<1, false>(L, A, G, P, d, p, B, T, k, ws, n_out, 0, 0, 0, s, launched,
                                nullptr, &test);
  return launch_cap<kMaxFusedLayers, false>(L, A, G, P, d, p, B, T, k, ws, n_out, 0, 0, 0, s,
                                            launched, nullptr, &test);
}

bool hutchpp12_planned(int64_t B, int64_t T, int64_t d, int64_t p) {
  HParams<kHppCap> a;
  const int64_t dd[2] = {d, p};
  const int64_t pp[2] = {p, d};
  int grid = 0;
  return plan_fused<kHppCap, false>(2, dd, pp, B, T, 32, a, grid);
}

cudaError_t launch_tc_hutchpp12(const void* A, const void* G, const void* SP, int64_t B,
                                int64_t T, int64_t d, int64_t p, const FusedScratch& ws, void* Z,
                                float* YP, float* M, void* MH, cudaStream_t s, bool* launched) {
  *launched = false;
  static thread_local HParams<kHppCap> a;
  // pass 1 projects onto the rows of d (A) and sketches p (G); pass 2 the
  // other way round
  const int64_t dd[2] = {d, p};
  const int64_t pp[2] = {p, d};
  int grid = 0;
  if (!plan_fused<kHppCap, false>(2, dd, pp, B, T, 32, a, grid)) return cudaSuccess;
  a.wait_ns = kWaitLimitNs;
  a.tpad = ws.tpad;
  // One sketch buffer serves both passes: pass 2's sketch of sample i starts
  // only once every pass-1 projection block of sample i has finished.
  for (int b = 0; b < 3; ++b) a.W[b] = static_cast<__nv_bfloat16*>(ws.W[0]);
  a.ready = ws.ready;
  a.tickets = ws.tickets;
  a.lticket = ws.lticket;
  a.done2 = ws.done2;
  a.exit_count = ws.exit_count;
  a.chunk_norms = ws.chunk_norms;
  a.nl = ws.nl;
  a.n_out = nullptr;
  a.accumulate = 0;
  a.norm_scale = 1.0f;
  a.clip_C = 0.f;
  a.c_out = nullptr;
  a.nonfinite = nullptr;
  a.seed = a.step = 0;
  a.hz = static_cast<__nv_bfloat16*>(Z);
  a.hyp = YP;
  a.hm = M;
  a.hmh = static_cast<__nv_bfloat16*>(MH);
  a.zdone = ws.lticket;
  a.zdone_target = a.layer[0].nchunks * (a.layer[0].ph2.split ? a.cl : 1);
  a.mdone_target = a.layer[1].nchunks * (a.layer[1].ph2.split ? a.cl : 1);
  for (int b = 0; b < 3; ++b)
    if (!make_tmap_3d_bf16(&a.mw[b], ws.W[0], T, 64, B, ws.tpad, 64 * ws.tpad, 64, 64, 128))
      return cudaErrorInvalidValue;
  LayerDesc& L0 = a.layer[0];
  LayerDesc& L1 = a.layer[1];
  if (!make_tmap_3d_bf16(&L0.mg, G, p, T, B, p, T * p, 64, kTok, 128) ||
      !make_tmap_3d_bf16(&L0.mp, SP, 32, p, 1, 32, p * 32, 32, kCol, 64) ||
      !make_tmap_3d_bf16(&L0.ma, A, d, T, B, d, T * d, 64, kTok, 128) ||
      !make_tmap_3d_bf16(&L1.mg, A, d, T, B, d, T * d, 64, kTok, 128) ||
      !make_tmap_3d_bf16(&L1.mp, Z, 32, d, B, 32, d * 32, 32, kCol, 64) ||
      !make_tmap_3d_bf16(&L1.ma, G, p, T, B, p, T * p, 64, kTok, 128))
    return cudaErrorInvalidValue;
  const cudaError_t e = launch_k<32, kHppCap, false>(a, grid, s);
  if (e == cudaSuccess) *launched = true;
  return e;
}

cudaError_t launch_tc_hutch_pm1(const void* A, const void* G, int64_t B, int64_t T, int64_t d,
                                int64_t p, int64_t k, uint64_t seed, uint64_t step,
                                const FusedScratch& ws, float* n_out, int accumulate,
                                cudaStream_t s, bool* launched) {
  *launched = false;
  const void* P = nullptr;
  return launch_cap<1, true>(1, &A, &G, &P, &d, &p, B, T, k, ws, n_out, accumulate, seed, step, s,
                             launched, nullptr);
}

}  // namespace dprc
