// Narrow layers (one width <= 64, e.g. the two maps of a low-rank adapter):
// the per-sample weight gradient itself is small, so it is formed once.
//
// "Efficient DP-SGD for LLMs with Randomized Clipping" (papernotes.org,
// "Key design > Hutchinson") sketches the d x p gradient A_i^T G_i with a
// p x k projection because forming it costs O(T d p) and its memory is d p
// per sample.  When min(d, p) <= 64 (adapters of rank 8..64: the notes run
// LoRA fine-tuning beside full fine-tuning, "Experiments") that product is no
// more work than the sketch, and X_i = A_i^T G_i arrives tile by tile in
// on-chip memory.  One streaming pass over A and G then gives
//
//   exact norm   n_i = ||X_i||_F^2                   (any orientation)
//   Hutchinson   n_i = scale ||X_i P||_F^2, p <= 64   (each row of X_i times P)
//
// the second equal to the sketch path's ||A_i^T (G_i P)||^2 up to rounding
// (the product is associative, and rows of X_i P depend on rows of X_i only).
// For the +-1 projection P = S, its p k signs are generated from the Philox
// stream into shared memory; S never exists in global memory.
//
// tc_narrow_kernel: tiles of 128 columns of the wide operand (the one whose
// width is > 64, or A when both are narrow) against all columns of the narrow
// operand, K = T in 64-token stages, accumulated in fp32 TMEM by tcgen05.mma.
// Both operands are MN-major, read as stored: the wide tile as two 64-column
// boxes with a 128-byte swizzle, the narrow one as one box N columns wide
// (N = 16, 32 or 64, the narrow width rounded up; the TMA fills the columns
// past it with zeros) with a 2N-byte swizzle.  A stage is 18 to 24 KB, so
// eight of them keep 144 to 192 KB per SM in flight.  The accumulator is
// double buffered.  The epilogue (one TMEM lane, i.e. one row of the tile, per
// thread) squares and sums the row, or first multiplies it by P (staged in
// shared memory in bf16; for p <= 16 on the tensor cores, the rows of X as
// bf16 hi/lo against P), and writes one partial per tile; the CTA that
// completes a sample's last tile (a per-sample ticket) adds the sample's
// partials in tile order: one launch, deterministic.

#include <atomic>
#include <type_traits>

#include "common.cuh"
#include "internal.h"

namespace dprc {

namespace {

constexpr int kNwM = 128;                    // wide columns per tile (MMA M)
constexpr int kNwK = 64;                     // tokens per stage
constexpr int kNwStages = 8;
constexpr int kNwBox = kNwK * 64 * 2;        // 64 tokens x 64 wide columns, 8 KB
constexpr int kNwWide = (kNwM / 64) * kNwBox;  // 16 KB

// Row stride (floats) of the tile's X rows in shared memory in the d-narrow
// estimate: a multiple of four, so each row starts on a 16-byte boundary.
__host__ __device__ constexpr int nx_of(int n) { return n + 4; }

template <int N>
struct NwCfg {
  static constexpr int kNarrow = kNwK * N * 2;       // 64 tokens x N narrow columns
  static constexpr int kStage = kNwWide + kNarrow;   // 18, 20 or 24 KB
  static constexpr int kTmemCols = 2 * N < 32 ? 32 : 2 * N;
  static constexpr int kCtrl = 256;
  static constexpr int kBase = 1024 + kNwStages * kStage + kCtrl;
  // P (bf16, at most 64 x 256) in shared memory after the barriers
  static constexpr int smem(int proj_bytes) { return kBase + proj_bytes; }
  static_assert(kStage % 1024 == 0, "stages keep the 1024-byte alignment of swizzled tiles");
};

// kNwNorm: ||rows||^2; kNwProj: ||row P||^2 (p narrow, rows = d);
// kNwProjT: the tile's part of X_i P (d narrow, rows = p), X_tile^T P_tile.
enum NwMode { kNwNorm = 0, kNwProj = 1, kNwProjT = 2 };

struct NwArgs {
  int T;
  int wide, narrow;   // widths of the wide and narrow operands
  int mt;             // wide tiles per sample
  long long ntiles;   // B * mt
  float* partials;    // [ntiles]
  // projection mode (the narrow operand is G, narrow = p):
  const void* P;      // [p][k] in the input type, or null for the +-1 signs
  int k, kp;          // kp: k rounded up to a multiple of 16 (shared-memory rows)
  float scale;
  uint64_t seed, step;  // the signs' Philox stream when P is null
  float* ypart;         // kNwProjT: [ntiles][narrow * k] partial products
  // the last tile of a sample adds its parts into n_out (tickets: zero on
  // entry, zero again on exit)
  int* tickets;         // [B]
  float* n_out;
  int accumulate;
  // optional clip factors of the final n_out (c_out non-null)
  float clip_C;
  float* c_out;
  int32_t* nonfinite;
};

// Copies `total` consecutive entries of a row-major [.][k] matrix into rows of
// kp entries in shared memory, by the 128 epilogue threads (index et), with
// four independent loads in flight per thread.
template <typename TP>
__device__ __forceinline__ void stage_rows(const TP* __restrict__ src, int total, int k, int kp,
                                           TP* dst, int et) {
  for (int e0 = et; e0 < total; e0 += 4 * 128) {
    TP v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + 128 * u;
      v[u] = e < total ? src[e] : static_cast<TP>(0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int e = e0 + 128 * u;
      if (e < total) dst[(e / k) * kp + e % k] = v[u];
    }
  }
}

// Outputs o = et + 128 m (m < nm <= NM) of a tile's part of X_i P when k
// divides 128: they share the column c = et % k and take rows
// a = et / k + m 128 / k of X; each is a sum over the tile's rows in order.
template <int NM, typename TP>
__device__ __forceinline__ void shared_col_outputs(const float* Xs, int nx, const TP* Pt, int kp,
                                                   int k, int rows, int et, int nm, float* dst) {
  const int c = et % k, a0 = et / k, astep = kNwM / k;
  float y[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) y[m] = 0.f;
  for (int r = 0; r < rows; ++r) {
    const float pv = static_cast<float>(Pt[r * kp + c]);
    const float* xr = Xs + r * nx + a0;
#pragma unroll
    for (int m = 0; m < NM; ++m)
      if (m < nm) y[m] = fmaf(xr[m * astep], pv, y[m]);
  }
  if (dst != nullptr) {
#pragma unroll
    for (int m = 0; m < NM; ++m)
      if (m < nm) dst[et + m * kNwM] = y[m];
  }
}

// A tile's part of X_i P (d narrow, rows = p indices) with the outputs in
// register blocks: thread et owns rows 4 dq .. 4 dq + 3 of X^T P against
// columns 2 kq, 2 kq + 1, over one of `parts` equal ranges of the tile's rows,
// so each row costs one 16-byte load of X and one 4-byte load of P for eight
// products, and the eight sums are independent.  Needs k even and
// (narrow / 4) (k / 2) dividing 128 (blocked_fits).  The parts are then added
// in part order through shared memory (Xs, once every thread is done with
// it) and the sums written row-major [narrow][k] to dst (skipped if null).
__device__ __forceinline__ bool blocked_fits(int narrow, int k) {
  if ((k & 1) != 0 || (narrow & 3) != 0) return false;
  const int items = (narrow >> 2) * (k >> 1);
  return items > 0 && kNwM % items == 0;
}

__device__ __forceinline__ void blocked_outputs(float* Xs, int nx, const __nv_bfloat16* Pt,
                                                int kp, int k, int narrow, int rows, int et,
                                                float* dst) {
  const int nk2 = k >> 1, items = (narrow >> 2) * nk2, parts = kNwM / items;
  const int h = et / items, it = et - h * items;
  const int dq = it / nk2, kq = it - dq * nk2;
  const int rlen = kNwM / parts;
  const int r0 = h * rlen, r1 = r0 + rlen < rows ? r0 + rlen : rows;
  float acc[4][2];
#pragma unroll
  for (int m = 0; m < 4; ++m) acc[m][0] = acc[m][1] = 0.f;
  auto row = [&](const float4& x, const float2& pv) {
    acc[0][0] = fmaf(x.x, pv.x, acc[0][0]);
    acc[0][1] = fmaf(x.x, pv.y, acc[0][1]);
    acc[1][0] = fmaf(x.y, pv.x, acc[1][0]);
    acc[1][1] = fmaf(x.y, pv.y, acc[1][1]);
    acc[2][0] = fmaf(x.z, pv.x, acc[2][0]);
    acc[2][1] = fmaf(x.z, pv.y, acc[2][1]);
    acc[3][0] = fmaf(x.w, pv.x, acc[3][0]);
    acc[3][1] = fmaf(x.w, pv.y, acc[3][1]);
  };
  // one warp per scheduler runs this, so nothing else hides the load
  // latency: eight rows' loads are issued before their products
  int r = r0;
  for (; r + 8 <= r1; r += 8) {
    float4 x[8];
    __nv_bfloat162 pb[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      x[u] = *reinterpret_cast<const float4*>(Xs + (r + u) * nx + 4 * dq);
      pb[u] = *reinterpret_cast<const __nv_bfloat162*>(Pt + (r + u) * kp + 2 * kq);
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) row(x[u], __bfloat1622float2(pb[u]));
  }
  for (; r < r1; ++r)
    row(*reinterpret_cast<const float4*>(Xs + r * nx + 4 * dq),
        __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(Pt + r * kp + 2 * kq)));
  named_bar_sync(1, 128);  // every part is done reading Xs
  if (h > 0) {
    float* red = Xs + ((h - 1) * items + it) * 8;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      red[2 * m] = acc[m][0];
      red[2 * m + 1] = acc[m][1];
    }
  }
  named_bar_sync(1, 128);
  if (h == 0 && dst != nullptr) {
    for (int hh = 1; hh < parts; ++hh) {
      const float* red = Xs + ((hh - 1) * items + it) * 8;
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        acc[m][0] += red[2 * m];
        acc[m][1] += red[2 * m + 1];
      }
    }
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      float* o = dst + (4 * dq + m) * k + 2 * kq;
      o[0] = acc[m][0];
      o[1] = acc[m][1];
    }
  }
}

// Rows [p0, p0 + rows) of P (or of the +-1 signs, entry e = r k + c of the
// Philox stream of (seed, step)) into Pt [128][kp], by the 128 epilogue
// threads.
template <typename TP, typename Args>
__device__ __forceinline__ void stage_p_tile(const Args& a, int p0, int rows, TP* Pt, int et) {
  if (a.P != nullptr) {
    // one contiguous run of P: coalesced loads, four in flight per thread
    stage_rows(static_cast<const TP*>(a.P) + static_cast<size_t>(p0) * a.k, rows * a.k, a.k,
               a.kp, Pt, et);
    return;
  }
  const RoundKeys rk = round_keys(a.seed);
  const long long e0 = static_cast<long long>(p0) * a.k;
  const long long e1 = e0 + static_cast<long long>(rows) * a.k;
  for (long long jb = e0 / 128 + et; jb * 128 < e1; jb += 128) {
    const uint4 w = philox_block(static_cast<uint64_t>(jb), a.step, rk);
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int wq = 0; wq < 4; ++wq)
      for (int b = 0; b < 32; ++b) {
        const long long e = jb * 128 + wq * 32 + b;
        if (e >= e0 && e < e1) {
          const int r = static_cast<int>((e - e0) / a.k);
          const int c = static_cast<int>((e - e0) - static_cast<long long>(r) * a.k);
          Pt[r * a.kp + c] = static_cast<TP>(((words[wq] >> b) & 1u) ? -1.0f : 1.0f);
        }
      }
  }
}

// p narrow (<= 16), kp = 16, 32 or 64: the rows of X_i P come from the tensor
// cores.  Each epilogue thread writes its row of X as bf16 hi and lo into two
// A tiles (128 rows x 16, K-major, 32-byte swizzle: 16-byte chunk c of row r
// at c ^ ((r >> 2) & 1)); P sits once per CTA in a B tile (16 rows x kp,
// MN-major, 2 kp-byte swizzle); one thread issues X_hi P and X_lo P into
// kp TMEM columns after the accumulators, and every thread squares its row of
// the product.
__host__ __device__ __forceinline__ bool rows_mma_fits(int N, int kp) {
  return N == 16 && (kp == 16 || kp == 32 || kp == 64);
}
constexpr int kNwRowsExtra = 1024 + 2048 + 2 * 4096;  // alignment, B tile, A tiles hi/lo
constexpr int kNwResCol = 32;                         // first TMEM column of X P

// chunk of a 16-byte chunk c in row r of a tile of `bytes`-wide swizzled rows
__device__ __forceinline__ int swz_chunk(int c, int r, int bytes) {
  return bytes == 128 ? (c ^ (r & 7)) : (bytes == 64 ? (c ^ ((r >> 1) & 3)) : (c ^ ((r >> 2) & 1)));
}

template <int KP>
__device__ __forceinline__ float rows_mma_square(uint32_t taddr) {
  float y[KP];
  tmem_ld_cols<KP>(taddr, y);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int c = 0; c < KP; c += 2) {
    s0 = fmaf(y[c], y[c], s0);
    s1 = fmaf(y[c + 1], y[c + 1], s1);
  }
  return s0 + s1;
}

template <int N, int MODE, typename TP>
__global__ void __launch_bounds__(192, 1)
    tc_narrow_kernel(const __grid_constant__ CUtensorMap map_w,
                     const __grid_constant__ CUtensorMap map_n, const NwArgs a) {
  using Cfg = NwCfg<N>;
  extern __shared__ uint8_t smem_raw[];
  __shared__ float s_red[4];
  __shared__ int s_last;
  __shared__ int s_live[4];

  uint8_t* ring = align_1024(smem_raw);
  TP* Ps = reinterpret_cast<TP*>(ring + kNwStages * Cfg::kStage + Cfg::kCtrl);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + kNwStages * Cfg::kStage);
  uint64_t* empty = full + kNwStages;
  uint64_t* accf = empty + kNwStages;  // [2]
  uint64_t* acce = accf + 2;           // [2]
  uint64_t* drain = acce + 2;          // MMA thread: all its MMAs complete
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acce + 3);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint64_t* pbar = acce + 4;           // the epilogue's X P products complete
  uint64_t* edrain = acce + 5;         // the epilogue's issuer: all its MMAs complete
  // the row products on tensor cores (kNwProj, p <= 16): TMEM for them too
  constexpr int kTmemAlloc = MODE == kNwProj && N == 16 ? 128 : Cfg::kTmemCols;
  const bool rows_mma = MODE == kNwProj && rows_mma_fits(N, a.kp);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nu = (a.T + kNwK - 1) / kNwK;  // stages per tile
  const long long my_tiles =
      a.ntiles > blockIdx.x ? (a.ntiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;

  // stage u of the tile at (sample i, wide tile m) into ring slot s.  Each
  // wide tile is read once, with the evict-first L2 policy; the narrow rows
  // are read again by every tile of the sample and keep the default.
  auto load_stage = [&](int i, int m, int u, int s) {
    uint8_t* st = ring + s * Cfg::kStage;
    mbar_arrive_expect_tx(&full[s], Cfg::kStage);
    const uint64_t pol = l2_policy_evict_first();
#pragma unroll
    for (int h = 0; h < kNwM / 64; ++h)
      tma_load_3d_hint(st + h * kNwBox, &map_w, &full[s], m * kNwM + h * 64, u * kNwK, i, pol);
    tma_load_3d(st + kNwWide, &map_n, &full[s], 0, u * kNwK, i);
  };
  // The launch is a programmatic dependent of the previous kernel in the
  // stream: the next launch may set up now, and this one's threads wait for
  // the previous grid's completion before they touch global memory (thread 0
  // before its first loads, the epilogue before P and its outputs).
  pdl_launch_dependents();
  // the producer (thread 0) issues the first stages of its first tile right
  // after initialising the barriers: their DRAM round trip overlaps the TMEM
  // allocation and the CTA barrier
  const int pre = my_tiles > 0 ? (nu < kNwStages ? nu : kNwStages) : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kNwStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&accf[b], 1);
      mbar_init(&acce[b], 4);
    }
    mbar_init(drain, 1);
    mbar_init(pbar, 1);
    mbar_init(edrain, 1);
    fence_mbar_init();
    *abort_flag = 0;
    const int i0 = static_cast<int>(blockIdx.x / a.mt);
    const int m0 = static_cast<int>(blockIdx.x - static_cast<long long>(i0) * a.mt);
    pdl_wait();
    for (int u = 0; u < pre; ++u) load_stage(i0, m0, u, u);
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&map_w);
    tma_prefetch_desc(&map_n);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kTmemAlloc);
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
        const int i = static_cast<int>(tile / a.mt);
        const int m = static_cast<int>(tile - static_cast<long long>(i) * a.mt);
        for (int u = 0; u < nu; ++u, ++it) {
          if (it < pre) continue;  // issued before the CTA barrier
          const int s = static_cast<int>(it % kNwStages);
          const uint32_t ph = static_cast<uint32_t>(it / kNwStages) & 1;
          if (!mbar_wait(&empty[s], ph ^ 1, DPRC_DEVERR_PIPE_EMPTY)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          load_stage(i, m, u, s);
        }
      }
      // let the copies this thread issued land before the CTA can exit
      for (long long k = it - 1; k >= 0 && k >= it - kNwStages; --k)
        mbar_wait(&full[k % kNwStages], (k / kNwStages) & 1, DPRC_DEVERR_PIPE_FULL);
    }
  } else if (warp == 1) {
    if (lane == 0 && my_tiles > 0) {
      constexpr uint32_t idesc = make_idesc_bf16(kNwM, N, true, true);
      constexpr uint32_t nswz = swz_code_for_bytes(2 * N);
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
          const int s = static_cast<int>(it % kNwStages);
          const uint32_t ph = static_cast<uint32_t>(it / kNwStages) & 1;
          if (!mbar_wait(&full[s], ph, DPRC_DEVERR_PIPE_FULL)) {
            *abort_flag = 1;
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t wa = smem_u32(ring + s * Cfg::kStage);
          const uint32_t na = wa + kNwWide;
#pragma unroll
          for (int kk = 0; kk < kNwK / 16; ++kk) {
            // wide tile: MN-major, 128-byte swizzle; a K = 16 step is 16 token
            // rows of 128 B, 8-row atoms 1 KB apart (SBO), the two 64-column
            // atoms one box apart (LBO)
            const uint64_t ad = make_sdesc(wa + kk * 2048, kNwBox, 1024, kSwz128);
            // narrow tile: MN-major, one swizzle atom wide (2N bytes); a K = 16
            // step is 16 rows of 2N bytes, 8-row atoms 16N bytes apart
            const uint64_t bd = make_sdesc(na + kk * 32 * N, 16, 16 * N, nswz);
            umma_bf16(tmem + abuf * N, ad, bd, idesc, (u == 0 && kk == 0) ? 0u : 1u);
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
    const int et = threadIdx.x - 64;
    pdl_wait();
    if (MODE == kNwProj) {
      // P (or the +-1 signs) into shared memory, once
      // rows of kp = k rounded up to 16 columns, zeros past k
      const int pk = a.narrow * a.k;
      for (int e = et; e < a.narrow * a.kp; e += 128) Ps[e] = static_cast<TP>(0.f);
      named_bar_sync(1, 128);
      if (a.P != nullptr) {
        stage_rows(static_cast<const TP*>(a.P), pk, a.k, a.kp, Ps, et);
      } else {
        // entry e of S: bit (e & 31) of word ((e >> 5) & 3) of block e >> 7
        const RoundKeys rk = round_keys(a.seed);
        for (int j = et; j * 128 < pk; j += 128) {
          const uint4 w = philox_block(static_cast<uint64_t>(j), a.step, rk);
          const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int wq = 0; wq < 4; ++wq)
            for (int b = 0; b < 32; ++b) {
              const int e = j * 128 + wq * 32 + b;
              if (e < pk)
                Ps[(e / a.k) * a.kp + e % a.k] =
                    static_cast<TP>(((words[wq] >> b) & 1u) ? -1.0f : 1.0f);
            }
        }
      }
      named_bar_sync(1, 128);
    }
    // the row products' tiles (rows_mma): B = P as 16 swizzled rows of kp,
    // then the A tiles of X hi and lo
    uint8_t* mbase = align_1024(reinterpret_cast<uint8_t*>(Ps) + 2048);
    uint8_t* PB = mbase;
    uint8_t* XAh = mbase + 2048;
    uint8_t* XAl = mbase + 2048 + 4096;
    if (rows_mma) {
      const int wb = 2 * a.kp, cpr = wb / 16;
      for (int e = et; e < 16 * cpr; e += 128) {
        const int b = e / cpr, c = e - b * cpr;
        uint4 v4 = make_uint4(0u, 0u, 0u, 0u);
        if (b < a.narrow) v4 = *reinterpret_cast<const uint4*>(Ps + b * a.kp + 8 * c);
        *reinterpret_cast<uint4*>(PB + b * wb + 16 * swz_chunk(c, b, wb)) = v4;
      }
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      named_bar_sync(1, 128);
    }
    uint32_t pphase = 0;    // parity of the next product batch
    bool e_issued = false;  // thread et 0 issued products (drained before exit)
    bool ok = true;
    for (long long j = 0; j < my_tiles; ++j) {
      const long long tile = blockIdx.x + j * gridDim.x;
      const int abuf = static_cast<int>(j & 1);
      if (MODE == kNwProjT) {
        // the tile's rows of P do not depend on X: staged while the MMAs run
        const int i = static_cast<int>(tile / a.mt);
        const int p0 = static_cast<int>(tile - static_cast<long long>(i) * a.mt) * kNwM;
        const int rows = a.wide - p0 < kNwM ? a.wide - p0 : kNwM;
        TP* Pt = reinterpret_cast<TP*>(reinterpret_cast<float*>(Ps) + kNwM * nx_of(N));
        stage_p_tile(a, p0, rows, Pt, et);
        named_bar_sync(1, 128);
      }
      bool live = ok && mbar_wait(&accf[abuf], static_cast<uint32_t>((j >> 1) & 1),
                                  DPRC_DEVERR_ACCUM) &&
                  *abort_flag == 0;
      live = __all_sync(0xffffffffu, live);  // keep the warp's TMEM loads convergent
      if (!live) ok = false;
      tc_fence_after();
      float v[N];
      if (live) {
        const uint32_t tb = tmem + (static_cast<uint32_t>(q * 32) << 16) + abuf * N;
#pragma unroll
        for (int c0 = 0; c0 < N; c0 += 16) {
          float t[16];
          tmem_ld_16cols(tb + c0, t);
#pragma unroll
          for (int c = 0; c < 16; ++c) v[c0 + c] = t[c];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce[abuf]);
      if (MODE == kNwProjT) {
        // rows of the tile are p indices p0 + r: the tile's part of X_i P is
        // sum_r x_r^T P[p0 + r] (d x k).  The rows go to shared memory (Xs,
        // fp32 [128][N + 1]) beside the tile's rows of P (Pt, staged above),
        // then each thread forms d k / 128 entries, each summed over r in
        // a fixed order.
        constexpr int NX = nx_of(N);  // rows 16-byte aligned
        float* Xs = reinterpret_cast<float*>(Ps);
        TP* Pt = reinterpret_cast<TP*>(Xs + kNwM * NX);
        const int i = static_cast<int>(tile / a.mt);
        const int p0 = static_cast<int>(tile - static_cast<long long>(i) * a.mt) * kNwM;
        const int rows = a.wide - p0 < kNwM ? a.wide - p0 : kNwM;
        const int row = q * 32 + lane;
#pragma unroll
        for (int c = 0; c < N; ++c) Xs[row * NX + c] = live ? v[c] : 0.f;
        named_bar_sync(1, 128);
        const bool lok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        const int dk = a.narrow * a.k;
        bool blocked = false;
        if constexpr (std::is_same<TP, __nv_bfloat16>::value) {
          if (blocked_fits(a.narrow, a.k)) {
            blocked_outputs(Xs, NX, Pt, a.kp, a.k, a.narrow, rows, et,
                            lok && DPRC_IN(tile < a.ntiles) ? a.ypart + tile * dk : nullptr);
            blocked = true;
          }
        }
        if (blocked) {
        } else if (kNwM % a.k == 0 && dk <= 32 * kNwM) {
          // k divides 128: this thread's outputs et + 128 m share the column
          // c = et % k, so each P element is loaded once per row
          const int nm = (dk - et + kNwM - 1) / kNwM;
          float* dst = lok && DPRC_IN(tile < a.ntiles) ? a.ypart + tile * dk : nullptr;
          if (nm <= 4)
            shared_col_outputs<4>(Xs, NX, Pt, a.kp, a.k, rows, et, nm, dst);
          else if (nm <= 8)
            shared_col_outputs<8>(Xs, NX, Pt, a.kp, a.k, rows, et, nm, dst);
          else if (nm <= 16)
            shared_col_outputs<16>(Xs, NX, Pt, a.kp, a.k, rows, et, nm, dst);
          else
            shared_col_outputs<32>(Xs, NX, Pt, a.kp, a.k, rows, et, nm, dst);
        } else {
          for (int o = et; o < dk; o += 128) {
            const int ad = o / a.k, c = o - (o / a.k) * a.k;
            // eight partial sums over r (r mod 8; rows is a multiple of 8),
            // added in a fixed order
            float y[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) y[u] = 0.f;
            for (int r = 0; r < rows; r += 8) {
#pragma unroll
              for (int u = 0; u < 8; ++u)
                y[u] = fmaf(Xs[(r + u) * NX + ad], static_cast<float>(Pt[(r + u) * a.kp + c]),
                            y[u]);
            }
            const float t = ((y[0] + y[1]) + (y[2] + y[3])) + ((y[4] + y[5]) + (y[6] + y[7]));
            if (lok && DPRC_IN(tile < a.ntiles)) a.ypart[tile * dk + o] = t;
          }
        }
        named_bar_sync(1, 128);  // Xs and Pt are rewritten by the next tile
      } else {
      float sq = 0.f;
      if (MODE == kNwProj && rows_mma) {
        // X row -> bf16 hi/lo A rows; every epilogue thread takes part in the
        // barriers, and the products are issued only if every warp is live
        const int row = q * 32 + lane;
        if (live) {
          uint32_t hw[8], lw[8];
#pragma unroll
          for (int t2 = 0; t2 < 8; ++t2) {
            __nv_bfloat16 h0, l0, h1, l1;
            split_hilo(v[2 * t2], h0, l0);
            split_hilo(v[2 * t2 + 1], h1, l1);
            const __nv_bfloat162 hh = __halves2bfloat162(h0, h1);
            const __nv_bfloat162 ll = __halves2bfloat162(l0, l1);
            hw[t2] = *reinterpret_cast<const uint32_t*>(&hh);
            lw[t2] = *reinterpret_cast<const uint32_t*>(&ll);
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int pc = swz_chunk(c, row, 32);
            *reinterpret_cast<uint4*>(XAh + row * 32 + 16 * pc) =
                make_uint4(hw[4 * c], hw[4 * c + 1], hw[4 * c + 2], hw[4 * c + 3]);
            *reinterpret_cast<uint4*>(XAl + row * 32 + 16 * pc) =
                make_uint4(lw[4 * c], lw[4 * c + 1], lw[4 * c + 2], lw[4 * c + 3]);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        if (lane == 0) s_live[ew] = live ? 1 : 0;
        named_bar_sync(1, 128);
        const bool go = s_live[0] && s_live[1] && s_live[2] && s_live[3];
        if (go) {
          if (et == 0) {
            tc_fence_after();
            const uint32_t idesc = make_idesc_bf16(128, a.kp, false, true);
            const uint64_t bd =
                make_sdesc(smem_u32(PB), 16, 16 * a.kp, swz_code_for_bytes(2 * a.kp));
            umma_bf16(tmem + kNwResCol, make_sdesc(smem_u32(XAh), 16, 256, kSwz32), bd, idesc, 0u);
            umma_bf16(tmem + kNwResCol, make_sdesc(smem_u32(XAl), 16, 256, kSwz32), bd, idesc, 1u);
            umma_commit(pbar);
            e_issued = true;
          }
          bool done = mbar_wait(pbar, pphase, DPRC_DEVERR_ACCUM);
          pphase ^= 1u;
          done = __all_sync(0xffffffffu, done);
          tc_fence_after();
          if (done) {
            const uint32_t tr = tmem + (static_cast<uint32_t>(q * 32) << 16) + kNwResCol;
            sq = a.kp == 16 ? rows_mma_square<16>(tr)
                            : (a.kp == 32 ? rows_mma_square<32>(tr) : rows_mma_square<64>(tr));
            sq *= a.scale;
          } else {
            ok = false;
          }
        }
        tc_fence_before();
        named_bar_sync(1, 128);  // the A tiles and the product columns are reused next tile
      } else if (live) {
        if (MODE == kNwNorm) {
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int c = 0; c < N; c += 2) {
            s0 = fmaf(v[c], v[c], s0);
            s1 = fmaf(v[c + 1], v[c + 1], s1);
          }
          sq = s0 + s1;
        } else {
          // ||x P||^2 for this row x (columns past p are zero), 16 columns of
          // x P at a time; every thread reads the same P entries (broadcast),
          // 8 bf16 per 16-byte load (P's rows are padded to kp columns)
          for (int c0 = 0; c0 < a.k; c0 += 16) {
            float y[16];
#pragma unroll
            for (int c = 0; c < 16; ++c) y[c] = 0.f;
#pragma unroll
            for (int b = 0; b < N; ++b) {
              if (b < a.narrow) {
                const uint4* pr = reinterpret_cast<const uint4*>(Ps + b * a.kp + c0);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                  const uint4 w = pr[h];
                  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                  for (int c2 = 0; c2 < 4; ++c2) {
                    const float lo = __uint_as_float(ws[c2] << 16);
                    const float hi = __uint_as_float(ws[c2] & 0xFFFF0000u);
                    y[8 * h + 2 * c2] = fmaf(v[b], lo, y[8 * h + 2 * c2]);
                    y[8 * h + 2 * c2 + 1] = fmaf(v[b], hi, y[8 * h + 2 * c2 + 1]);
                  }
                }
              }
            }
#pragma unroll
            for (int c = 0; c < 16; ++c) sq = fmaf(y[c], y[c], sq);
          }
          sq *= a.scale;
        }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, off);
      if (lane == 0) s_red[ew] = sq;
      named_bar_sync(1, 128);
      if (ew == 0 && lane == 0 && ok && DPRC_IN(tile < a.ntiles))
        a.partials[tile] = (s_red[0] + s_red[1]) + (s_red[2] + s_red[3]);
      named_bar_sync(1, 128);
      }  // MODE != kNwProjT
      // the CTA that completes a sample's last tile adds the sample's parts,
      // in tile order, into n_out
      const int is = static_cast<int>(tile / a.mt);
      __threadfence();  // this thread's partial writes, before the ticket
      named_bar_sync(1, 128);
      if (et == 0)
        s_last = DPRC_IN(tile < a.ntiles) && atomicAdd(&a.tickets[is], 1) == a.mt - 1;
      named_bar_sync(1, 128);
      if (s_last) {
        __threadfence();
        float acc = 0.f;
        if (MODE == kNwProjT) {
          // entry e of the sample's X_i P is the sum over its tiles m, in m
          // order; four entries at a time, sixteen tiles per batch of loads, so
          // 64 loads are in flight (this runs at the very end of the launch)
          const int dk = a.narrow * a.k;
          const float* yi = a.ypart + static_cast<size_t>(is) * a.mt * dk;
          for (int e0 = et; e0 < dk; e0 += 4 * 128) {
            float y[4] = {0.f, 0.f, 0.f, 0.f};
            for (int m = 0; m < a.mt; m += 16) {
              float t[16][4];
#pragma unroll
              for (int u = 0; u < 16; ++u)
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2) {
                  const int e = e0 + q2 * 128;
                  t[u][q2] = (m + u < a.mt && e < dk)
                                 ? __ldcg(yi + static_cast<size_t>(m + u) * dk + e)
                                 : 0.f;
                }
#pragma unroll
              for (int u = 0; u < 16; ++u)
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2)
                  if (m + u < a.mt) y[q2] += t[u][q2];
            }
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) acc = fmaf(y[q2], y[q2], acc);
          }
          acc *= a.scale;
        } else if (ew == 0) {
          for (int m = lane; m < a.mt; m += 32)
            acc += __ldcg(a.partials + static_cast<size_t>(is) * a.mt + m);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) s_red[ew] = acc;
        named_bar_sync(1, 128);
        if (et == 0) {
          const float tot = (s_red[0] + s_red[1]) + (s_red[2] + s_red[3]);
          const float nv = (a.accumulate ? a.n_out[is] : 0.f) + tot;
          a.n_out[is] = nv;
          a.tickets[is] = 0;
          if (a.c_out != nullptr) {
            bool bad;
            a.c_out[is] = clip_factor(nv, a.clip_C, bad);
            if (bad && a.nonfinite != nullptr) atomicAdd(a.nonfinite, 1);
          }
        }
        named_bar_sync(1, 128);
      }
    }
    // the products this thread issued are complete before the TMEM is freed
    // (after a failed wait above they may still run)
    if (e_issued) umma_drain(edrain, kWaitLimitNs);
  }

  __syncwarp();  // reconverge each warp before the CTA barrier
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemAlloc);
  }
}

template <int N, int MODE, typename TP>
cudaError_t launch_n(const CUtensorMap& mw, const CUtensorMap& mn, const NwArgs& a,
                     int proj_bytes, cudaStream_t s) {
  auto kern = tc_narrow_kernel<N, MODE, TP>;
  constexpr int kMaxDev = 64;
  static std::atomic<int> done[kMaxDev];  // largest shared-memory size set so far
  const int smem = NwCfg<N>::smem(proj_bytes);
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDev || done[dev].load(std::memory_order_acquire) < smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDev) done[dev].store(smem, std::memory_order_release);
  }
  const long long grid = a.ntiles < device_sm_count() ? a.ntiles : device_sm_count();
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(192);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr.val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mw, mn, a);
}

template <int MODE, typename TP>
cudaError_t launch_mode(int N, const CUtensorMap& mw, const CUtensorMap& mn, const NwArgs& a,
                        int proj_bytes, cudaStream_t s) {
  return N == 16 ? launch_n<16, MODE, TP>(mw, mn, a, proj_bytes, s)
                 : (N == 32 ? launch_n<32, MODE, TP>(mw, mn, a, proj_bytes, s)
                            : launch_n<64, MODE, TP>(mw, mn, a, proj_bytes, s));
}

// Operands of X = A^T G as (wide, narrow): A is the wide one unless only d
// is narrow.
bool narrow_setup(const void* A, const void* G, int64_t B, int64_t T, int64_t d, int64_t p,
                  CUtensorMap& mw, CUtensorMap& mn, NwArgs& a, int& N) {
  const bool swap = d <= 64 && p > 64;
  const void* W = swap ? G : A;
  const void* Nr = swap ? A : G;
  const int64_t wide = swap ? p : d, narrow = swap ? d : p;
  N = narrow <= 16 ? 16 : (narrow <= 32 ? 32 : 64);
  if (!make_tmap_3d_bf16(&mw, W, wide, T, B, wide, T * wide, 64, kNwK, 128)) return false;
  if (!make_tmap_3d_bf16(&mn, Nr, narrow, T, B, narrow, T * narrow, N, kNwK, 2 * N))
    return false;
  a.T = static_cast<int>(T);
  a.wide = static_cast<int>(wide);
  a.narrow = static_cast<int>(narrow);
  a.mt = static_cast<int>((wide + kNwM - 1) / kNwM);
  a.ntiles = B * a.mt;
  a.partials = nullptr;
  a.P = nullptr;
  a.k = a.kp = 0;
  a.scale = 1.f;
  a.seed = a.step = 0;
  a.ypart = nullptr;
  a.tickets = nullptr;
  a.n_out = nullptr;
  a.accumulate = 0;
  a.clip_C = 0.f;
  a.c_out = nullptr;
  a.nonfinite = nullptr;
  return true;
}

}  // namespace

cudaError_t read_device_error_narrow(int32_t* out, bool reset) {
  return read_tu_device_error(out, reset);
}

bool narrow_supported(dprc_dtype dt, int64_t d, int64_t p) {
  return dt == DPRC_BF16 && d % 8 == 0 && p % 8 == 0 && (d <= 64 || p <= 64);
}

bool narrow_proj_supported(dprc_dtype dt, int64_t d, int64_t p, int64_t k) {
  if (dt != DPRC_BF16 || d % 8 != 0 || p % 8 != 0 || k < 1) return false;
  // rows of X_i P from rows of X_i (p narrow), or per-tile parts of it (d
  // narrow: the tile's rows and P's rows in shared memory next to the ring)
  return (p <= 64 && k <= 256) || (d <= 32 && p > 64 && k <= 128);
}

int64_t narrow_partials(int64_t B, int64_t d, int64_t p) {
  const int64_t wide = d <= 64 && p > 64 ? p : d;
  return B * ((wide + kNwM - 1) / kNwM);
}

size_t narrow_hutch_scratch_bytes(int64_t B, int64_t d, int64_t p, int64_t k) {
  const bool swap = d <= 64 && p > 64;
  const int64_t per = swap ? d * k : 1;  // floats per tile
  return static_cast<size_t>(narrow_partials(B, d, p) * per) * 4;
}

cudaError_t launch_narrow_norm(const void* A, const void* G, int64_t B, int64_t T, int64_t d,
                               int64_t p, int* tickets, float* partials, float* n_out,
                               int accumulate, cudaStream_t s) {
  CUtensorMap mw, mn;
  NwArgs a;
  int N = 16;
  if (!narrow_setup(A, G, B, T, d, p, mw, mn, a, N)) return cudaErrorInvalidValue;
  a.partials = partials;
  a.tickets = tickets;
  a.n_out = n_out;
  a.accumulate = accumulate;
  return launch_mode<kNwNorm, float>(N, mw, mn, a, 0, s);
}

cudaError_t launch_narrow_hutch(const void* A, const void* G, const void* P, int64_t B,
                                int64_t T, int64_t d, int64_t p, int64_t k, float scale,
                                uint64_t seed, uint64_t step, int* tickets, float* partials,
                                float* n_out, int accumulate, cudaStream_t s,
                                const ClipOut* clip) {
  if (!narrow_proj_supported(DPRC_BF16, d, p, k)) return cudaErrorInvalidValue;
  CUtensorMap mw, mn;
  NwArgs a;
  int N = 16;
  if (!narrow_setup(A, G, B, T, d, p, mw, mn, a, N)) return cudaErrorInvalidValue;
  a.P = P;
  a.k = static_cast<int>(k);
  a.kp = static_cast<int>((k + 15) / 16 * 16);
  a.scale = scale;
  a.seed = seed;
  a.step = step;
  a.tickets = tickets;
  a.n_out = n_out;
  a.accumulate = accumulate;
  if (clip != nullptr) {
    a.clip_C = clip->C;
    a.c_out = clip->c;
    a.nonfinite = clip->nonfinite;
  }
  if (p <= 64) {
    a.partials = partials;
    int proj_bytes = static_cast<int>(p * a.kp * 2);
    // P's rows for the CUDA-core product, or (p <= 16) room for the tensor
    // cores' tiles after them
    if (rows_mma_fits(N, a.kp)) proj_bytes = (proj_bytes > 2048 ? proj_bytes : 2048) + kNwRowsExtra;
    return launch_mode<kNwProj, __nv_bfloat16>(N, mw, mn, a, proj_bytes, s);
  }
  // d narrow: per-tile parts of X_i P (scratch: narrow_hutch_scratch_bytes)
  a.ypart = partials;
  const int proj_bytes = kNwM * nx_of(N) * 4 + kNwM * a.kp * 2;
  return launch_mode<kNwProjT, __nv_bfloat16>(N, mw, mn, a, proj_bytes, s);
}

}  // namespace dprc
