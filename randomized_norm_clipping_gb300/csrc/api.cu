// libdprc C ABI: argument checks, scratch layout, dispatch to the kernels.
//
// Data flow of one Hutchinson call (tensor-core path):
//   K1 row projection    W = G P             reads G once   (HBM-bound)
//   K2 column projection Y = A^T W, ||Y||^2  reads A once   (HBM-bound)
// K2 is launched with programmatic dependent launch so its prologue overlaps
// the tail of K1.  Hutch++ chains three such pairs with the per-sample QR in
// the middle; the float32 path runs the same steps on CUDA cores.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "dprc.h"
#include "internal.h"

namespace dprc {
namespace {

constexpr int kDefaultSms = 152;
constexpr int64_t kMaxT = int64_t(1) << 24;
constexpr int64_t kMaxWidth = int64_t(1) << 20;
constexpr int64_t kMaxB = 65535;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

dprc_status cuda_status(cudaError_t e) { return e == cudaSuccess ? DPRC_OK : DPRC_ERR_CUDA; }

// Per-thread optional events recorded between the kernels of a call (timing).
thread_local void** t_events = nullptr;
thread_local int t_nevents = 0;

void mark(int idx, cudaStream_t s) {
  if (t_events != nullptr && idx < t_nevents && t_events[idx] != nullptr)
    cudaEventRecord(static_cast<cudaEvent_t>(t_events[idx]), s);
}

constexpr int kMaxDev = 64;
std::atomic<int> g_dev_state[kMaxDev];  // 0 unknown, 1 sm_103, 2 other
std::atomic<int> g_dev_sms[kMaxDev];

// True if the current device is an sm_103 GPU (checked once per device).
bool device_ok() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (dev >= 0 && dev < kMaxDev) {
    const int st = g_dev_state[dev].load(std::memory_order_acquire);
    if (st != 0) return st == 1;
  }
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return false;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return false;
  const bool ok = major == 10 && minor == 3;
  if (dev >= 0 && dev < kMaxDev) g_dev_state[dev].store(ok ? 1 : 2, std::memory_order_release);
  return ok;
}

int64_t tpad_of(int64_t T) { return (T + 63) / 64 * 64; }

}  // namespace

int device_sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return kDefaultSms;
  if (dev >= 0 && dev < kMaxDev) {
    const int c = g_dev_sms[dev].load(std::memory_order_acquire);
    if (c > 0) return c;
  }
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
    return kDefaultSms;
  if (dev >= 0 && dev < kMaxDev) g_dev_sms[dev].store(n, std::memory_order_release);
  return n;
}

BlockSched make_block_sched(int64_t nblocks, int upb, int slots) {
  BlockSched s;
  s.nblocks = nblocks;
  s.upb = upb;
  if (nblocks * 4 >= static_cast<int64_t>(slots) * 3) {
    // enough blocks to fill the GPU: whole blocks, as evenly as possible
    s.cl = 1;
    s.bpc = static_cast<int>((nblocks + slots - 1) / slots);
    s.grid = static_cast<int>((nblocks + s.bpc - 1) / s.bpc);
  } else {
    // few blocks: split each across a cluster (power of two up to 8)
    s.cl = 1;
    while (s.cl < 8 && nblocks * s.cl * 2 <= slots && s.cl * 2 <= upb) s.cl *= 2;
    s.bpc = 1;
    s.grid = static_cast<int>(nblocks * s.cl);
  }
  return s;
}

BlockSched rowproj_sched(int64_t B, int64_t T, int64_t c, int nmma) {
  (void)nmma;
  return make_block_sched(B * ((T + 127) / 128), static_cast<int>((c + 63) / 64),
                          device_sm_count() * rowproj_ctas_per_sm());
}

BlockSched colproj_sched(int64_t B, int64_t T, int64_t c, int nmma) {
  const int64_t nch = (c + colproj_stage_chunk() - 1) / colproj_stage_chunk();
  return make_block_sched(B * nch, static_cast<int>((T + colproj_tile_t() - 1) / colproj_tile_t()),
                          device_sm_count() * colproj_ctas_per_sm(nmma));
}

bool tc_path_supported(dprc_dtype dt, int64_t B, int64_t T, int64_t d, int64_t p, int64_t k,
                       bool hutchpp) {
  (void)B;
  (void)T;
  if (dt != DPRC_BF16) return false;
  if (d % 8 != 0 || p % 8 != 0) return false;  // TMA row strides: multiples of 16 bytes
  if (hutchpp) return k == 16 && p >= k;
  return k == 16 || k == 32 || k == 64;
}

// Every plan starts with the same counter block: tickets and sketch-ready
// counters per (layer slot, sample), layers finished per sample, projection
// blocks finished per layer slot, and one CTA-exit count.  Calls leave it
// zeroed; the fused Hutchinson kernel relies on that, so no other buffer may
// overlap it.  Where the counters sit inside the block depends on B, so the
// block has one size for every B up to kCtrlFixedB: a call with fewer samples
// must not place its scratch where a call with more keeps counters (one
// workspace then serves calls with any B up to that bound).
constexpr int64_t kCtrlFixedB = 256;
size_t ctrl_bytes(int64_t B) {
  const int64_t Bc = B > kCtrlFixedB ? B : kCtrlFixedB;
  const size_t ints = 2 * static_cast<size_t>(kMaxFusedLayers) * Bc + Bc + kMaxFusedLayers + 1;
  return align_up(ints * 4, 256);
}

TcPlan plan_tc(dprc_op op, int64_t B, int64_t T, int64_t d, int64_t p, int64_t k, int layers) {
  TcPlan t;
  t.tpad = tpad_of(T);
  const int64_t nch = (std::max(d, p) + colproj_stage_chunk() - 1) / colproj_stage_chunk();
  const size_t LB = static_cast<size_t>(kMaxFusedLayers) * B;
  t.stick_off = 0;
  t.ready_off = LB * 4;
  t.lticket_off = 2 * LB * 4;
  t.done2_off = t.lticket_off + static_cast<size_t>(B) * 4;
  t.exit_off = t.done2_off + static_cast<size_t>(kMaxFusedLayers) * 4;
  size_t off = ctrl_bytes(B);
  t.cnorm_off = off;
  off = align_up(off + static_cast<size_t>(layers) * B * nch * 4, 1024);
  t.nl_off = off;
  off = align_up(off + static_cast<size_t>(layers) * B * 4, 1024);
  t.w_bytes = static_cast<size_t>(B) * (op == DPRC_OP_HUTCH ? 2 * k : 4 * k) * t.tpad * 2;
  t.w_off = off;
  off = align_up(off + t.w_bytes, 1024);
  t.w2_off = t.w3_off = t.w_off;
  if (layers > 1) {
    t.w2_off = off;
    off = align_up(off + t.w_bytes, 1024);
    t.w3_off = off;
    off = align_up(off + t.w_bytes, 1024);
  }
  if (op == DPRC_OP_HUTCHPP) {
    const int64_t r = k;
    t.z_off = off;
    off = align_up(off + static_cast<size_t>(B) * d * 2 * r * 2, 1024);
    t.m_off = off;
    off = align_up(off + static_cast<size_t>(B) * p * r * 4, 1024);
    t.qp_off = off;
    off = align_up(off + static_cast<size_t>(B) * p * 4 * r * 2, 1024);
    t.qscratch_off = off;
    off = align_up(off + static_cast<size_t>(B) * p * r * 4 * 2, 1024);
    t.sp_off = off;
    off = align_up(off + static_cast<size_t>(p) * 2 * r * 2, 1024);
    t.yp_off = off;
    off = align_up(off + static_cast<size_t>(B) * d * r * 4, 1024);
    t.rc_off = off;
    off = align_up(off + static_cast<size_t>(B) * qr_factor_floats() * 4, 1024);
  }
  t.total = off;
  return t;
}

FusedScratch fused_scratch(const TcPlan& t, char* w) {
  FusedScratch f;
  f.W[0] = w + t.w_off;
  f.W[1] = w + t.w2_off;
  f.W[2] = w + t.w3_off;
  f.tpad = t.tpad;
  f.tickets = reinterpret_cast<int*>(w + t.stick_off);
  f.ready = reinterpret_cast<int*>(w + t.ready_off);
  f.lticket = reinterpret_cast<int*>(w + t.lticket_off);
  f.done2 = reinterpret_cast<int*>(w + t.done2_off);
  f.exit_count = reinterpret_cast<int*>(w + t.exit_off);
  f.chunk_norms = reinterpret_cast<float*>(w + t.cnorm_off);
  f.nl = reinterpret_cast<float*>(w + t.nl_off);
  return f;
}

SimtPlan plan_simt(dprc_op op, int64_t B, int64_t T, int64_t d, int64_t p, int64_t k) {
  SimtPlan s;
  const int64_t wide = op == DPRC_OP_HUTCHPP ? 2 * k : k;
  size_t off = ctrl_bytes(B);
  s.w_off = off;
  off = align_up(off + static_cast<size_t>(B) * T * wide * 4, 1024);
  s.y_off = off;
  off = align_up(off + static_cast<size_t>(B) * d * wide * 4, 1024);
  if (op == DPRC_OP_HUTCHPP) {
    s.z_off = off;
    off = align_up(off + static_cast<size_t>(B) * d * k * 4, 1024);
    s.m_off = off;
    off = align_up(off + static_cast<size_t>(B) * p * k * 4, 1024);
    s.qp_off = off;
    off = align_up(off + static_cast<size_t>(B) * p * 2 * k * 4, 1024);
    s.qscratch_off = off;
    off = align_up(off + static_cast<size_t>(B) * p * k * 4 * 2, 1024);
  }
  s.total = off;
  return s;
}

// Tensor-core layout of the exact norm: bf16 with rows of d and p 16-byte
// multiples (TMA).  Both exact forms run there; other layouts take the ghost
// form on CUDA cores.
bool exact_direct_tc(dprc_dtype dt, int64_t d, int64_t p) {
  return dt == DPRC_BF16 && d % 8 == 0 && p % 8 == 0;
}

size_t exact_partials_off(int64_t B) { return align_up(ctrl_bytes(B), 1024); }

namespace {
// Longest T the tensor-core ghost form takes (its partials grow as T^2).
constexpr int64_t kGhostTcMaxT = 65536;
// Longest T of the CUDA-core ghost form (its grid has T / 32 rows).
constexpr int64_t kGhostSimtMaxT = int64_t(65535) * 32;

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Time of a persistent one-CTA-per-SM launch in units of one 128 x 256 x 64
// MMA stage of the ghost kernel, for the busiest CTA.  Direct form:
// B ceil(d/128) ceil(p/256) equal tiles of ceil(T/64) stages, dealt out with
// a stride of the grid.  Ghost form: B S_W(nt) units of (d + p) / 64 stages;
// a unit's time does not depend on its width (a 128 x 128 MMA takes about as
// long as a 128 x 256 one on this part), so the busiest CTA runs
// ceil(units / SMs) of them.  Relative stage rates measured on GB300: the
// direct kernel's stage 1.06, a 128 x 128 ghost stage 0.92 of a 128 x 256 one.
double exact_cost_direct(int64_t B, int64_t T, int64_t d, int64_t p, int sms) {
  const int64_t tiles = B * cdiv(d, 128) * cdiv(p, 256);
  return static_cast<double>(cdiv(tiles, sms)) * static_cast<double>(cdiv(T, 64)) * 1.06;
}

double exact_cost_ghost(int64_t B, int64_t T, int64_t d, int64_t p, int W, int sms) {
  const int64_t units = ghost_partials(B, T, W);
  const double stages = static_cast<double>(cdiv(d, 64) + cdiv(p, 64));
  return static_cast<double>(cdiv(units, sms)) * stages * (W == 1 ? 0.92 : 1.0);
}
}  // namespace

ExactPlan plan_exact(dprc_dtype dt, int64_t B, int64_t T, int64_t d, int64_t p, int form) {
  ExactPlan e;
  if (form < DPRC_EXACT_AUTO || form > DPRC_EXACT_GHOST_N256) return e;
  if (!exact_direct_tc(dt, d, p)) {
    if (form == DPRC_EXACT_DIRECT || form == DPRC_EXACT_GHOST_N128 ||
        form == DPRC_EXACT_GHOST_N256 || T > kGhostSimtMaxT)
      return e;
    e.kind = ExactPlan::kGhostSimt;
    e.per_sample = cdiv(T, 32) * cdiv(T, 32);
    return e;
  }
  if (form != DPRC_EXACT_GHOST && form != DPRC_EXACT_GHOST_N128 &&
      form != DPRC_EXACT_GHOST_N256 && narrow_supported(dt, d, p)) {
    // one width <= 64: the direct form in one pass, no tile padding (and
    // always less work than the ghost form's T^2 (d + p) when T >= 128)
    e.kind = ExactPlan::kNarrowTc;
    e.per_sample = narrow_partials(1, d, p);
    return e;
  }
  const int sms = device_sm_count() > 0 ? device_sm_count() : 1;
  const double cd = exact_cost_direct(B, T, d, p, sms);
  double cg = -1.0;
  int wg = 2;
  if (T <= kGhostTcMaxT) {
    const double c1 = exact_cost_ghost(B, T, d, p, 1, sms);
    const double c2 = exact_cost_ghost(B, T, d, p, 2, sms);
    wg = form == DPRC_EXACT_GHOST_N128 ? 1 : (form == DPRC_EXACT_GHOST_N256 ? 2 : (c1 < c2 ? 1 : 2));
    cg = wg == 1 ? c1 : c2;
  }
  const bool ghost = form == DPRC_EXACT_GHOST || form == DPRC_EXACT_GHOST_N128 ||
                     form == DPRC_EXACT_GHOST_N256 ||
                     (form == DPRC_EXACT_AUTO && cg >= 0 && cg < cd);
  if (ghost) {
    if (cg < 0) return e;
    e.kind = ExactPlan::kGhostTc;
    e.W = wg;
    e.per_sample = ghost_partials(1, T, wg);
  } else {
    e.kind = ExactPlan::kDirectTc;
    e.per_sample = fgc_partials(1, d, p);
  }
  return e;
}

size_t plan_exact_bytes(dprc_dtype dt, int64_t B, int64_t T, int64_t d, int64_t p) {
  // room for whichever form and span width a call takes (W = 1 has the most
  // ghost units), independent of the device
  int64_t most = 0;
  if (exact_direct_tc(dt, d, p)) {
    most = fgc_partials(1, d, p);
    if (narrow_supported(dt, d, p)) most = std::max(most, narrow_partials(1, d, p));
    if (T <= kGhostTcMaxT) most = std::max(most, ghost_partials(1, T, 1));
  } else {
    most = cdiv(T, 32) * cdiv(T, 32);
  }
  return exact_partials_off(B) + align_up(static_cast<size_t>(B) * most * 4, 1024);
}

// ---- tensor maps ------------------------------------------------------------
namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = []() -> EncodeTiledFn {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}
}  // namespace

bool make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1,
                       uint64_t dim2, uint64_t stride1_elems, uint64_t stride2_elems,
                       uint32_t box0, uint32_t box1, int swizzle_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[3] = {dim0, dim1, dim2};
  const cuuint64_t strides[2] = {stride1_elems * 2, stride2_elems * 2};
  const cuuint32_t box[3] = {box0, box1, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_NONE;
  if (swizzle_bytes == 32) swz = CU_TENSOR_MAP_SWIZZLE_32B;
  if (swizzle_bytes == 64) swz = CU_TENSOR_MAP_SWIZZLE_64B;
  if (swizzle_bytes == 128) swz = CU_TENSOR_MAP_SWIZZLE_128B;
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace dprc

using namespace dprc;

namespace {

dprc_status check_common(dprc_dtype dt, int64_t B, int64_t T, int64_t d, int64_t p) {
  if (dt != DPRC_F32 && dt != DPRC_BF16) return DPRC_ERR_DTYPE;
  if (B < 1 || T < 1 || d < 1 || p < 1) return DPRC_ERR_SHAPE;
  if (B > kMaxB || T > kMaxT || d > kMaxWidth || p > kMaxWidth) return DPRC_ERR_SHAPE;
  return DPRC_OK;
}

// Narrow layers keep their per-tile partials after the counter block.
size_t narrow_part_off(int64_t B) { return align_up(ctrl_bytes(B), 1024); }
size_t narrow_ws(int64_t B, int64_t d, int64_t p, int64_t k) {
  return narrow_part_off(B) + align_up(narrow_hutch_scratch_bytes(B, d, p, k), 1024);
}

size_t hutch_ws(dprc_dtype dt, int64_t B, int64_t T, int64_t d, int64_t p, int64_t k) {
  const size_t base = tc_path_supported(dt, B, T, d, p, k, false)
                          ? plan_tc(DPRC_OP_HUTCH, B, T, d, p, k).total
                          : plan_simt(DPRC_OP_HUTCH, B, T, d, p, k).total;
  return narrow_proj_supported(dt, d, p, k) ? std::max(base, narrow_ws(B, d, p, k)) : base;
}

size_t hutchpp_ws(dprc_dtype dt, int64_t B, int64_t T, int64_t d, int64_t p, int64_t r) {
  return tc_path_supported(dt, B, T, d, p, r, true) ? plan_tc(DPRC_OP_HUTCHPP, B, T, d, p, r).total
                                              : plan_simt(DPRC_OP_HUTCHPP, B, T, d, p, r).total;
}


// Sketch and projection as separate kernels (tensor cores for bf16 with
// aligned widths and k in {16, 32, 64}, CUDA cores otherwise), with the
// squared columns of Y weighted 1 for the first n_head and w_tail after.
cudaError_t hutch_kernels(const void* A, const void* G, const void* P, dprc_dtype dtype, int64_t B,
                          int64_t T, int64_t d, int64_t p, int64_t k, float* n, int accumulate,
                          char* w, int n_head, float w_tail, cudaStream_t s) {
  const int ik = static_cast<int>(k);
  if (tc_path_supported(dtype, B, T, d, p, k, false)) {
    const TcPlan t = plan_tc(DPRC_OP_HUTCH, B, T, d, p, k);
    int* stick = reinterpret_cast<int*>(w + t.stick_off);
    float* cnorm = reinterpret_cast<float*>(w + t.cnorm_off);
    cudaError_t e = launch_tc_rowproj(G, B, T, p, P, false, ik, false, w + t.w_off, t.tpad,
                                      rowproj_sched(B, T, p, ik), stick, B, s);
    if (e != cudaSuccess) return e;
    mark(1, s);
    e = launch_tc_colproj(A, B, T, d, w + t.w_off, t.tpad, ik, colproj_sched(B, T, d, 2 * ik),
                          stick, cnorm, kColprojNorm, n, accumulate, n_head, w_tail, nullptr,
                          nullptr, t_events == nullptr, s);
    mark(2, s);
    return e;
  }
  const SimtPlan sp = plan_simt(DPRC_OP_HUTCH, B, T, d, p, k);
  float* W = reinterpret_cast<float*>(w + sp.w_off);
  float* Y = reinterpret_cast<float*>(w + sp.y_off);
  cudaError_t e = launch_simt_rowproj(G, dtype, B, T, p, P, dtype, false, ik, W, s);
  if (e != cudaSuccess) return e;
  mark(1, s);
  e = launch_simt_colproj(A, dtype, B, T, d, W, ik, Y, s);
  if (e != cudaSuccess) return e;
  e = launch_simt_norm_finish(Y, B, d, ik, n_head, w_tail, n, accumulate, s);
  mark(2, s);
  return e;
}

// Workspace of dprc_norm_hutch_pm1: the Hutchinson plan, then room for S.
size_t pm1_ws(dprc_dtype dt, int64_t B, int64_t T, int64_t d, int64_t p, int64_t k) {
  return align_up(hutch_ws(dt, B, T, d, p, k), 1024) +
         align_up(static_cast<size_t>(p) * k * (dt == DPRC_F32 ? 4 : 2), 1024);
}

// Device buffer of dprc_norm_hutch_clip_host: the workspace of one chunk's
// call, the per-chunk n and c (16-byte aligned per chunk), P, and two slots
// that each hold one chunk of samples of A and G.  A chunk is the fewest
// samples that make at least 128 MB of A and G: fewer, larger copies keep the
// host link busy (each copy costs a few microseconds of set-up), while the
// kernel of the last chunk is all that does not hide under a copy.
struct HostStage {
  int64_t chunk = 0, nchunks = 0, pitch = 0;  // samples per chunk; n/c floats per chunk
  size_t ws_off = 0, ws_bytes = 0, n_off = 0, c_off = 0, p_off = 0;
  size_t rest_ws_off = 0, rest_ws_bytes = 0;  // the last chunk's own workspace when it is short
  size_t slot_off[2] = {0, 0}, a_bytes = 0, g_bytes = 0, total = 0;
};

HostStage plan_host_stage(dprc_dtype dt, int64_t B, int64_t T, int64_t d, int64_t p, int64_t k) {
  HostStage h;
  const size_t eb = dt == DPRC_F32 ? 4 : 2;
  const size_t sample = static_cast<size_t>(T) * (d + p) * eb;
  const size_t want = size_t(128) << 20;
  h.chunk = std::min<int64_t>(B, static_cast<int64_t>((want + sample - 1) / sample));
  h.nchunks = (B + h.chunk - 1) / h.chunk;
  h.pitch = (h.chunk + 3) / 4 * 4;
  h.ws_bytes = hutch_ws(dt, h.chunk, T, d, p, k);
  size_t off = 0;
  h.ws_off = off;
  off = align_up(off + h.ws_bytes, 1024);
  // a shorter last chunk gets a workspace of its own: its counter block and
  // scratch are laid out for another B, and a workspace is shared only by
  // calls whose counter blocks coincide
  const int64_t rest = B % h.chunk;
  if (rest > 0) {
    h.rest_ws_bytes = hutch_ws(dt, rest, T, d, p, k);
    h.rest_ws_off = off;
    off = align_up(off + h.rest_ws_bytes, 1024);
  }
  h.n_off = off;
  off = align_up(off + static_cast<size_t>(h.nchunks) * h.pitch * 4, 1024);
  h.c_off = off;
  off = align_up(off + static_cast<size_t>(h.nchunks) * h.pitch * 4, 1024);
  h.p_off = off;
  off = align_up(off + static_cast<size_t>(p) * k * eb, 1024);
  h.a_bytes = static_cast<size_t>(h.chunk) * T * d * eb;
  h.g_bytes = static_cast<size_t>(h.chunk) * T * p * eb;
  for (int sl = 0; sl < 2; ++sl) {
    h.slot_off[sl] = off;
    off = align_up(off + align_up(h.a_bytes, 1024) + h.g_bytes, 1024);
  }
  h.total = off;
  return h;
}

// Two copy streams per device for the host-input entry (A and G of a chunk
// travel side by side, so one copy's set-up overlaps the other's transfer),
// created on first use.
constexpr int kMaxCopyDev = 64;
cudaStream_t g_copy_stream[kMaxCopyDev][2];
std::mutex g_copy_mu;

cudaStream_t copy_stream(int which) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxCopyDev) return nullptr;
  std::lock_guard<std::mutex> lock(g_copy_mu);
  cudaStream_t& cs = g_copy_stream[dev][which];
  if (cs == nullptr && cudaStreamCreateWithFlags(&cs, cudaStreamNonBlocking) != cudaSuccess)
    cs = nullptr;
  return cs;
}

}  // namespace

namespace dprc {
dprc_status check_hutch_args(const void* A, const void* G, const void* P, dprc_dtype dtype,
                             int64_t B, int64_t T, int64_t d, int64_t p, int64_t k,
                             const float* n) {
  if (!A || !G || !P || !n) return DPRC_ERR_NULL;
  const dprc_status st = check_common(dtype, B, T, d, p);
  if (st != DPRC_OK) return st;
  if (k < 1 || k > 256) return DPRC_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(G) || !aligned16(P) || !aligned16(n)) return DPRC_ERR_ALIGN;
  return DPRC_OK;
}

bool current_device_supported() { return device_ok(); }
}  // namespace dprc

namespace {
// dprc_norm_hutch, with the clip factors of the updated n when `clip` is set
// (in the fused kernel's finishing step, else by the clip kernel afterwards).
dprc_status norm_hutch_impl(const void* A, const void* G, const void* P, dprc_dtype dtype,
                            int64_t B, int64_t T, int64_t d, int64_t p, int64_t k, float* n,
                            int accumulate, void* ws, size_t ws_bytes, void* stream,
                            const ClipOut* clip) {
  const dprc_status st = check_hutch_args(A, G, P, dtype, B, T, d, p, k, n);
  if (st != DPRC_OK) return st;
  if (clip != nullptr) {
    if (!clip->c) return DPRC_ERR_NULL;
    if (!(clip->C > 0.f) || !(clip->C < __builtin_inff())) return DPRC_ERR_SHAPE;
    if (!aligned16(clip->c)) return DPRC_ERR_ALIGN;
  }
  if (!ws) return DPRC_ERR_WORKSPACE;
  if (!aligned16(ws)) return DPRC_ERR_ALIGN;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  if (ws_bytes < hutch_ws(dtype, B, T, d, p, k)) return DPRC_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  auto clip_after = [&](cudaError_t e) -> dprc_status {
    if (e == cudaSuccess && clip != nullptr) e = launch_clip(n, B, clip->C, clip->c, clip->nonfinite, s);
    return cuda_status(e);
  };
  mark(0, s);
  if (narrow_proj_supported(dtype, d, p, k)) {
    // a width <= 64: X_i = A_i^T G_i in one pass, times P in the epilogue
    // (and the clip factors in the same launch)
    const cudaError_t e =
        launch_narrow_hutch(A, G, P, B, T, d, p, k, 1.0f, 0, 0, reinterpret_cast<int*>(w),
                            reinterpret_cast<float*>(w + narrow_part_off(B)), n, accumulate, s,
                            clip);
    mark(1, s);
    mark(2, s);
    return cuda_status(e);
  }
  if (tc_path_supported(dtype, B, T, d, p, k, false) && fused_hutch_supported(k)) {
    // one launch: sketch and projection as two phases of one kernel (and the
    // clip factors in its finishing step)
    const TcPlan t = plan_tc(DPRC_OP_HUTCH, B, T, d, p, k);
    bool launched = false;
    const cudaError_t e = launch_tc_hutch_layers(1, &A, &G, &P, &d, &p, B, T, k,
                                                 fused_scratch(t, w), n, accumulate, s, &launched,
                                                 clip);
    if (launched) {
      mark(1, s);
      mark(2, s);
      return cuda_status(e);
    }
    if (e != cudaSuccess) (void)cudaGetLastError();  // not launched: two kernels below
  }
  return clip_after(hutch_kernels(A, G, P, dtype, B, T, d, p, k, n, accumulate, w,
                                  static_cast<int>(k), 1.0f, s));
}
}  // namespace

namespace {
// dprc_norm_hutch_layers, with the clip factors of the final layer sum when
// `clip` is set (in the launch that adds the last layer).
dprc_status norm_hutch_layers_impl(int64_t L, const void* const* A, const void* const* G,
                                   const void* const* P, const int64_t* d, const int64_t* p,
                                   dprc_dtype dtype, int64_t B, int64_t T, int64_t k, float* n,
                                   int accumulate, void* ws, size_t ws_bytes, void* stream,
                                   const ClipOut* clip) {
  if (!A || !G || !P || !d || !p || !n) return DPRC_ERR_NULL;
  if (clip != nullptr) {
    if (!clip->c) return DPRC_ERR_NULL;
    if (!(clip->C > 0.f) || !(clip->C < __builtin_inff())) return DPRC_ERR_SHAPE;
    if (!aligned16(clip->c)) return DPRC_ERR_ALIGN;
  }
  if (L < 1 || L > (int64_t(1) << 20)) return DPRC_ERR_SHAPE;
  if (k < 1 || k > 256) return DPRC_ERR_SHAPE;
  int64_t dmax = 0, pmax = 0;
  bool fused = fused_hutch_supported(k);
  for (int64_t l = 0; l < L; ++l) {
    if (!A[l] || !G[l] || !P[l]) return DPRC_ERR_NULL;
    const dprc_status st = check_common(dtype, B, T, d[l], p[l]);
    if (st != DPRC_OK) return st;
    if (!aligned16(A[l]) || !aligned16(G[l]) || !aligned16(P[l])) return DPRC_ERR_ALIGN;
    dmax = std::max(dmax, d[l]);
    pmax = std::max(pmax, p[l]);
    fused = fused && tc_path_supported(dtype, B, T, d[l], p[l], k, false);
  }
  if (!aligned16(n)) return DPRC_ERR_ALIGN;
  if (!ws) return DPRC_ERR_WORKSPACE;
  if (!aligned16(ws)) return DPRC_ERR_ALIGN;
  if (ws_bytes < dprc_workspace_bytes(DPRC_OP_HUTCH_LAYERS, dtype, B, T, dmax, pmax, k))
    return DPRC_ERR_WORKSPACE;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int64_t l0 = 0;
  if (fused) {
    const TcPlan t = plan_tc(DPRC_OP_HUTCH, B, T, dmax, pmax, k, kMaxFusedLayers);
    const FusedScratch f = fused_scratch(t, static_cast<char*>(ws));
    for (; l0 < L; l0 += kMaxFusedLayers) {
      const int Lc = static_cast<int>(std::min<int64_t>(kMaxFusedLayers, L - l0));
      bool launched = false;
      const cudaError_t e = launch_tc_hutch_layers(Lc, A + l0, G + l0, P + l0, d + l0, p + l0, B,
                                                   T, k, f, n, accumulate || l0 > 0, s,
                                                   &launched, l0 + Lc == L ? clip : nullptr);
      if (!launched) {
        if (e != cudaSuccess) (void)cudaGetLastError();
        break;  // the remaining layers one call at a time
      }
    }
  }
  for (int64_t l = l0; l < L; ++l) {
    const dprc_status st = norm_hutch_impl(A[l], G[l], P[l], dtype, B, T, d[l], p[l], k, n,
                                           accumulate || l > 0, ws, ws_bytes, stream,
                                           l == L - 1 ? clip : nullptr);
    if (st != DPRC_OK) return st;
  }
  return DPRC_OK;
}
}  // namespace



extern "C" {

int dprc_abi_version(void) { return DPRC_ABI_VERSION; }

const char* dprc_status_string(dprc_status s) {
  switch (s) {
    case DPRC_OK: return "ok";
    case DPRC_ERR_NULL: return "null pointer argument";
    case DPRC_ERR_SHAPE: return "size out of range or inconsistent";
    case DPRC_ERR_DTYPE: return "unknown dtype";
    case DPRC_ERR_ALIGN: return "pointer not 16-byte aligned";
    case DPRC_ERR_WORKSPACE: return "workspace missing or too small";
    case DPRC_ERR_CUDA: return "CUDA call failed";
    case DPRC_ERR_NONFINITE: return "non-finite value";
    case DPRC_ERR_DEVICE: return "current device is not an sm_103 GPU";
    case DPRC_ERR_TOO_LARGE: return "call needs more scratch than the built-in buffer";
  }
  return "unknown status";
}

size_t dprc_workspace_bytes(dprc_op op, dprc_dtype dtype, int64_t B, int64_t T, int64_t d,
                            int64_t p, int64_t k) {
  if (check_common(dtype, B, T, d, p) != DPRC_OK) return 0;
  switch (op) {
    case DPRC_OP_HUTCH:
      if (k < 1 || k > 256) return 0;
      return hutch_ws(dtype, B, T, d, p, k);
    case DPRC_OP_HUTCHPP:
      if (k < 1 || k > 64 || k > p) return 0;
      return hutchpp_ws(dtype, B, T, d, p, k);
    case DPRC_OP_EXACT:
      return plan_exact_bytes(dtype, B, T, d, p);
    case DPRC_OP_HUTCH_PM1:
      if (k < 1 || k > 256) return 0;
      return pm1_ws(dtype, B, T, d, p, k);
    case DPRC_OP_HUTCH_HOST:
      if (k < 1 || k > 256) return 0;
      return plan_host_stage(dtype, B, T, d, p, k).total;
    case DPRC_OP_HUTCH_LAYERS: {
      if (k < 1 || k > 256) return 0;
      // any layer with widths up to (d, p), including narrow ones taken one
      // call at a time
      size_t w = std::max(hutch_ws(dtype, B, T, d, p, k),
                          plan_tc(DPRC_OP_HUTCH, B, T, d, p, k, kMaxFusedLayers).total);
      w = std::max(w, narrow_ws(B, std::min<int64_t>(d, 32), p, k));
      w = std::max(w, narrow_ws(B, d, std::min<int64_t>(p, 64), k));
      return w;
    }
  }
  return 0;
}

dprc_status dprc_set_phase_events(void** events, int n_events) {
  if (n_events < 0 || (n_events > 0 && events == nullptr)) return DPRC_ERR_NULL;
  t_events = n_events > 0 ? events : nullptr;
  t_nevents = n_events;
  return DPRC_OK;
}


dprc_status dprc_norm_hutch(const void* A, const void* G, const void* P, dprc_dtype dtype,
                            int64_t B, int64_t T, int64_t d, int64_t p, int64_t k, float* n,
                            int accumulate, void* ws, size_t ws_bytes, void* stream) {
  DPRC_NVTX_RANGE();
  return norm_hutch_impl(A, G, P, dtype, B, T, d, p, k, n, accumulate, ws, ws_bytes, stream,
                         nullptr);
}

dprc_status dprc_norm_hutch_layers(int64_t L, const void* const* A, const void* const* G,
                                   const void* const* P, const int64_t* d, const int64_t* p,
                                   dprc_dtype dtype, int64_t B, int64_t T, int64_t k, float* n,
                                   int accumulate, void* ws, size_t ws_bytes, void* stream) {
  DPRC_NVTX_RANGE();
  return norm_hutch_layers_impl(L, A, G, P, d, p, dtype, B, T, k, n, accumulate, ws, ws_bytes,
                                stream, nullptr);
}

dprc_status dprc_norm_hutch_layers_clip(int64_t L, const void* const* A, const void* const* G,
                                        const void* const* P, const int64_t* d, const int64_t* p,
                                        dprc_dtype dtype, int64_t B, int64_t T, int64_t k,
                                        float* n, int accumulate, float C, float* c,
                                        int32_t* nonfinite, void* ws, size_t ws_bytes,
                                        void* stream) {
  DPRC_NVTX_RANGE();
  ClipOut clip;
  clip.C = C;
  clip.c = c;
  clip.nonfinite = nonfinite;
  return norm_hutch_layers_impl(L, A, G, P, d, p, dtype, B, T, k, n, accumulate, ws, ws_bytes,
                                stream, &clip);
}

dprc_status dprc_norm_hutch_clip(const void* A, const void* G, const void* P, dprc_dtype dtype,
                                 int64_t B, int64_t T, int64_t d, int64_t p, int64_t k, float* n,
                                 int accumulate, float C, float* c, int32_t* nonfinite, void* ws,
                                 size_t ws_bytes, void* stream) {
  DPRC_NVTX_RANGE();
  ClipOut clip;
  clip.C = C;
  clip.c = c;
  clip.nonfinite = nonfinite;
  return norm_hutch_impl(A, G, P, dtype, B, T, d, p, k, n, accumulate, ws, ws_bytes, stream,
                         &clip);
}

dprc_status dprc_norm_hutch_clip_host(const void* A, const void* G, const void* P,
                                      dprc_dtype dtype, int64_t B, int64_t T, int64_t d,
                                      int64_t p, int64_t k, float C, float* n, float* c,
                                      void* stage, size_t stage_bytes, void* stream) {
  DPRC_NVTX_RANGE();
  if (!A || !G || !P || !c) return DPRC_ERR_NULL;
  dprc_status st = check_common(dtype, B, T, d, p);
  if (st != DPRC_OK) return st;
  if (k < 1 || k > 256) return DPRC_ERR_SHAPE;
  if (!(C > 0.f) || !(C < __builtin_inff())) return DPRC_ERR_SHAPE;
  if (!stage) return DPRC_ERR_WORKSPACE;
  if (!aligned16(stage)) return DPRC_ERR_ALIGN;
  const HostStage h = plan_host_stage(dtype, B, T, d, p, k);
  if (stage_bytes < h.total) return DPRC_ERR_WORKSPACE;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaStream_t cs[2] = {copy_stream(0), copy_stream(1)};
  if (cs[0] == nullptr || cs[1] == nullptr) return DPRC_ERR_CUDA;
  char* w = static_cast<char*>(stage);
  const size_t eb = dtype == DPRC_F32 ? 4 : 2;
  float* nd = reinterpret_cast<float*>(w + h.n_off);
  float* cd = reinterpret_cast<float*>(w + h.c_off);
  void* Pd = w + h.p_off;
  // events: [0] start; per slot: A copied, G copied, slot free again
  constexpr int kEv = 7;
  cudaEvent_t ev[kEv] = {};
  cudaError_t e = cudaSuccess;
  for (int q = 0; q < kEv && e == cudaSuccess; ++q)
    e = cudaEventCreateWithFlags(&ev[q], cudaEventDisableTiming);
  cudaEvent_t start = ev[0];
  auto copied = [&](int operand, int sl) { return ev[1 + 2 * sl + operand]; };
  auto freed = [&](int sl) { return ev[5 + sl]; };
  // the copies follow the work already on the caller's stream (which may use
  // the stage buffer); chunk j's copies wait until the kernels of chunk j - 2
  // are done with its slot; chunk j's kernels wait for both copies
  if (e == cudaSuccess) e = cudaEventRecord(start, s);
  for (int q = 0; q < 2 && e == cudaSuccess; ++q) e = cudaStreamWaitEvent(cs[q], start, 0);
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(Pd, P, static_cast<size_t>(p) * k * eb, cudaMemcpyHostToDevice, cs[1]);
  for (int64_t j = 0; j < h.nchunks && e == cudaSuccess && st == DPRC_OK; ++j) {
    const int sl = static_cast<int>(j & 1);
    const int64_t i0 = j * h.chunk;
    const int64_t bc = std::min<int64_t>(h.chunk, B - i0);
    char* Ad = w + h.slot_off[sl];
    char* Gd = Ad + align_up(h.a_bytes, 1024);
    for (int q = 0; q < 2 && e == cudaSuccess; ++q) {
      const int64_t wq = q == 0 ? d : p;
      if (j >= 2) e = cudaStreamWaitEvent(cs[q], freed(sl), 0);
      if (e == cudaSuccess)
        e = cudaMemcpyAsync(q == 0 ? Ad : Gd,
                            static_cast<const char*>(q == 0 ? A : G) +
                                static_cast<size_t>(i0) * T * wq * eb,
                            static_cast<size_t>(bc) * T * wq * eb, cudaMemcpyHostToDevice, cs[q]);
      if (e == cudaSuccess) e = cudaEventRecord(copied(q, sl), cs[q]);
      if (e == cudaSuccess) e = cudaStreamWaitEvent(s, copied(q, sl), 0);
    }
    if (e != cudaSuccess) break;
    ClipOut clip;
    clip.C = C;
    clip.c = cd + j * h.pitch;
    const bool short_chunk = bc < h.chunk;
    st = norm_hutch_impl(Ad, Gd, Pd, dtype, bc, T, d, p, k, nd + j * h.pitch, 0,
                         w + (short_chunk ? h.rest_ws_off : h.ws_off),
                         short_chunk ? h.rest_ws_bytes : h.ws_bytes, s, &clip);
    if (st == DPRC_OK) e = cudaEventRecord(freed(sl), s);
  }
  // n and c back to the host: chunk j's values sit at j * pitch
  const int64_t full = B / h.chunk, rest = B - full * h.chunk;
  for (int q = n ? 0 : 1; q < 2 && e == cudaSuccess && st == DPRC_OK; ++q) {
    float* dst = q == 0 ? n : c;
    const float* src = q == 0 ? nd : cd;
    if (full > 0)
      e = cudaMemcpy2DAsync(dst, static_cast<size_t>(h.chunk) * 4, src,
                            static_cast<size_t>(h.pitch) * 4, static_cast<size_t>(h.chunk) * 4,
                            static_cast<size_t>(full), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess && rest > 0)
      e = cudaMemcpyAsync(dst + full * h.chunk, src + full * h.pitch,
                          static_cast<size_t>(rest) * 4, cudaMemcpyDeviceToHost, s);
  }
  // (events are released once the work recorded on them completes)
  for (int q = 0; q < kEv; ++q)
    if (ev[q]) cudaEventDestroy(ev[q]);
  if (st != DPRC_OK) return st;
  return cuda_status(e);
}

dprc_status dprc_norm_hutch_pm1(const void* A, const void* G, uint64_t seed, uint64_t step,
                                dprc_dtype dtype, int64_t B, int64_t T, int64_t d, int64_t p,
                                int64_t k, float* n, int accumulate, void* ws, size_t ws_bytes,
                                void* stream) {
  DPRC_NVTX_RANGE();
  if (!A || !G || !n) return DPRC_ERR_NULL;
  dprc_status st = check_common(dtype, B, T, d, p);
  if (st != DPRC_OK) return st;
  if (k < 1 || k > 256) return DPRC_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(G) || !aligned16(n)) return DPRC_ERR_ALIGN;
  if (!ws) return DPRC_ERR_WORKSPACE;
  if (!aligned16(ws)) return DPRC_ERR_ALIGN;
  if (ws_bytes < pm1_ws(dtype, B, T, d, p, k)) return DPRC_ERR_WORKSPACE;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  if (narrow_proj_supported(dtype, d, p, k)) {
    // a width <= 64: X_i = A_i^T G_i in one pass, then (1/k) ||X_i S||^2
    // with the signs generated in the kernel's shared memory
    return cuda_status(launch_narrow_hutch(A, G, nullptr, B, T, d, p, k,
                                           1.0f / static_cast<float>(k), seed, step,
                                           reinterpret_cast<int*>(w),
                                           reinterpret_cast<float*>(w + narrow_part_off(B)), n,
                                           accumulate, s));
  }
  if (tc_path_supported(dtype, B, T, d, p, k, false) && fused_hutch_supported(k)) {
    // the signs are generated inside the kernel: S never exists in memory
    const TcPlan t = plan_tc(DPRC_OP_HUTCH, B, T, d, p, k);
    bool launched = false;
    const cudaError_t e = launch_tc_hutch_pm1(A, G, B, T, d, p, k, seed, step, fused_scratch(t, w),
                                              n, accumulate, s, &launched);
    if (launched) return cuda_status(e);
    if (e != cudaSuccess) (void)cudaGetLastError();
  }
  // other shapes: the signs into the workspace, then the usual kernels with
  // every column weighted 1/k
  char* S = w + align_up(hutch_ws(dtype, B, T, d, p, k), 1024);
  cudaError_t e = launch_pm1_signs(S, dtype, p * k, seed, step, s);
  if (e != cudaSuccess) return DPRC_ERR_CUDA;
  return cuda_status(hutch_kernels(A, G, S, dtype, B, T, d, p, k, n, accumulate, w, 0,
                                   1.0f / static_cast<float>(k), s));
}

int dprc_norm_hutch_launches(dprc_dtype dtype, int64_t B, int64_t T, int64_t d, int64_t p,
                             int64_t k) {
  if (check_common(dtype, B, T, d, p) != DPRC_OK || k < 1 || k > 256) return 0;
  if (!device_ok()) return 0;
  if (narrow_proj_supported(dtype, d, p, k)) return 1;
  if (!tc_path_supported(dtype, B, T, d, p, k, false)) return 3;
  return fused_hutch_planned(B, T, d, p, k) ? 1 : 2;
}

int dprc_norm_hutchpp_launches(dprc_dtype dtype, int64_t B, int64_t T, int64_t d, int64_t p,
                               int64_t r) {
  if (check_common(dtype, B, T, d, p) != DPRC_OK || r < 1 || r > 64 || r > p) return 0;
  if (!device_ok()) return 0;
  if (!tc_path_supported(dtype, B, T, d, p, r, true)) return 8;
  if (!qr_cluster_supported(p, static_cast<int>(r))) return 7;
  return hutchpp12_planned(B, T, d, p) ? 5 : 8;
}

dprc_status dprc_norm_hutchpp(const void* A, const void* G, const void* S, const void* P,
                              dprc_dtype dtype, int64_t B, int64_t T, int64_t d, int64_t p,
                              int64_t r, float* n, int accumulate, void* ws, size_t ws_bytes,
                              void* stream) {
  DPRC_NVTX_RANGE();
  if (!A || !G || !S || !P || !n) return DPRC_ERR_NULL;
  dprc_status st = check_common(dtype, B, T, d, p);
  if (st != DPRC_OK) return st;
  if (r < 1 || r > 64 || r > p) return DPRC_ERR_SHAPE;
  if (!aligned16(A) || !aligned16(G) || !aligned16(S) || !aligned16(P) || !aligned16(n))
    return DPRC_ERR_ALIGN;
  if (!ws) return DPRC_ERR_WORKSPACE;
  if (!aligned16(ws)) return DPRC_ERR_ALIGN;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  char* w = static_cast<char*>(ws);
  const int ir = static_cast<int>(r);
  if (tc_path_supported(dtype, B, T, d, p, r, true)) {
    const TcPlan t = plan_tc(DPRC_OP_HUTCHPP, B, T, d, p, r);
    if (ws_bytes < t.total) return DPRC_ERR_WORKSPACE;
    int* stick = reinterpret_cast<int*>(w + t.stick_off);
    float* cnorm = reinterpret_cast<float*>(w + t.cnorm_off);
    void* W = w + t.w_off;
    void* Z = w + t.z_off;
    float* M = reinterpret_cast<float*>(w + t.m_off);
    void* QP = w + t.qp_off;
    const bool pdl = t_events == nullptr;
    if (qr_cluster_supported(p, ir)) {
      // the QR runs beside the third pass, which streams X M instead of X Q
      // (hutchpp.cu): X Q = (X M) diag(s) R^-1, X P' = X P - (X Q) C
      void* SP = w + t.sp_off;
      float* YP = reinterpret_cast<float*>(w + t.yp_off);
      float* RC = reinterpret_cast<float*>(w + t.rc_off);
      void* MH = QP;  // M as bf16 hi/lo [B][p][2r], the third pass's sketch operand
      // Each projection streams a sample as soon as the sample's sketch is
      // written (per-sample counts, rows 1, 2 and 0 of the block of counts for
      // passes 1, 2 and 3) instead of after the sketch kernel's end; only its
      // epilogue waits for that end.  The third pass's last blocks zero all three.
      int* ready = pdl ? reinterpret_cast<int*>(w + t.ready_off) : nullptr;
      int* ready1 = ready ? ready + B : nullptr;
      int* ready2 = ready ? ready + 2 * B : nullptr;
      const int ready_target = static_cast<int>((T + 127) / 128);
      mark(0, s);
      cudaError_t e = launch_pack_cols(S, P, SP, p, ir, s);
      // passes 1 and 2 as one persistent launch of the fused kernel (pass 2's
      // sketch of a sample starts when pass 1 has written that sample's Z)
      bool fused12 = false;
      if (e == cudaSuccess && pdl)
        e = launch_tc_hutchpp12(A, G, SP, B, T, d, p, fused_scratch(t, w), Z, YP, M, MH, s,
                                &fused12);
      if (e == cudaSuccess && !fused12) {
        // pass 1: [Z | X P] = A^T (G [S | P]); Z as hi/lo for pass 2, X P in fp32
        const BlockSched rs1 = rowproj_sched(B, T, p, 2 * ir);
        e = launch_tc_rowproj(G, B, T, p, SP, false, 2 * ir, false, W, t.tpad, rs1, stick, B, s,
                              false, ready1);
        if (e == cudaSuccess)
          e = launch_tc_colproj(A, B, T, d, W, t.tpad, 2 * ir, colproj_sched(B, T, d, 4 * ir),
                                stick, cnorm, kColprojSplit, nullptr, 0, ir, 1.0f, YP, Z, pdl, s,
                                ir, nullptr, nullptr, ready1, ready_target * rs1.cl);
        mark(1, s);
        // pass 2: M = G^T (A Z) = O S, fp32 for the QR and hi/lo for pass 3
        const BlockSched rs2 = rowproj_sched(B, T, d, 2 * ir);
        if (e == cudaSuccess)
          e = launch_tc_rowproj(A, B, T, d, Z, true, 2 * ir, true, W, t.tpad, rs2, stick, B, s,
                                false, ready2);
        if (e == cudaSuccess)
          e = launch_tc_colproj(G, B, T, p, W, t.tpad, ir, colproj_sched(B, T, p, 2 * ir), stick,
                                cnorm, kColprojF32Hilo, nullptr, 0, ir, 1.0f, M, MH, pdl, s, 0,
                                nullptr, nullptr, ready2, ready_target * rs2.cl);
      }
      mark(2, s);
      // the QR's factors (R, column scales, C = Q^T P) ...
      if (e == cudaSuccess) e = launch_qr_cluster(M, B, p, P, dtype, nullptr, true, s, RC);
      mark(3, s);
      // ... while pass 3 streams X M = A^T (G M); its epilogue forms
      // n (+)= ||X Q||^2 + ||X P'||^2 / r row by row from X M, X P and them
      // (the sketch kernel's end waits for the QR)
      const BlockSched rs3 = rowproj_sched(B, T, p, 2 * ir);
      if (e == cudaSuccess)
        e = launch_tc_rowproj(G, B, T, p, MH, true, 2 * ir, true, W, t.tpad, rs3, stick, B, s,
                              pdl, ready);
      if (e == cudaSuccess)
        e = launch_tc_colproj(A, B, T, d, W, t.tpad, ir, colproj_sched(B, T, d, 2 * ir), stick,
                              cnorm, kColprojHpp, n, accumulate, ir, 1.0f, nullptr, nullptr, pdl,
                              s, 0, RC, YP, ready, ready_target * rs3.cl, 3);
      mark(4, s);
      return cuda_status(e);
    }
    mark(0, s);
    // pass 1: Z = A^T (G S)
    cudaError_t e = launch_tc_rowproj(G, B, T, p, S, false, ir, false, W, t.tpad,
                                      rowproj_sched(B, T, p, ir), stick, B, s);
    if (e == cudaSuccess)
      e = launch_tc_colproj(A, B, T, d, W, t.tpad, ir, colproj_sched(B, T, d, 2 * ir), stick,
                            cnorm, kColprojHilo, nullptr, 0, ir, 1.0f, nullptr, Z, pdl, s);
    mark(1, s);
    // pass 2: M = G^T (A Z) = O S
    if (e == cudaSuccess)
      e = launch_tc_rowproj(A, B, T, d, Z, true, 2 * ir, true, W, t.tpad,
                            rowproj_sched(B, T, d, 2 * ir), stick, B, s);
    if (e == cudaSuccess)
      e = launch_tc_colproj(G, B, T, p, W, t.tpad, ir, colproj_sched(B, T, p, 2 * ir), stick,
                            cnorm, kColprojF32, nullptr, 0, ir, 1.0f, M, nullptr, pdl, s);
    mark(2, s);
    // Q = qr(M), P' = P - Q Q^T P
    if (e == cudaSuccess)
      e = launch_qr_project(M, B, p, ir, P, dtype,
                            reinterpret_cast<float*>(w + t.qscratch_off), QP, true, s);
    mark(3, s);
    // pass 3: Y = A^T G [Q | P'], n = ||Y_head||^2 + ||Y_tail||^2 / r
    if (e == cudaSuccess)
      e = launch_tc_rowproj(G, B, T, p, QP, true, 4 * ir, true, W, t.tpad,
                            rowproj_sched(B, T, p, 4 * ir), stick, B, s);
    if (e == cudaSuccess)
      e = launch_tc_colproj(A, B, T, d, W, t.tpad, 2 * ir, colproj_sched(B, T, d, 4 * ir), stick,
                            cnorm, kColprojNorm, n, accumulate, ir, 1.0f / static_cast<float>(r),
                            nullptr, nullptr, pdl, s);
    mark(4, s);
    return cuda_status(e);
  }
  const SimtPlan sp = plan_simt(DPRC_OP_HUTCHPP, B, T, d, p, r);
  if (ws_bytes < sp.total) return DPRC_ERR_WORKSPACE;
  float* W = reinterpret_cast<float*>(w + sp.w_off);
  float* Y = reinterpret_cast<float*>(w + sp.y_off);
  float* Z = reinterpret_cast<float*>(w + sp.z_off);
  float* M = reinterpret_cast<float*>(w + sp.m_off);
  float* QP = reinterpret_cast<float*>(w + sp.qp_off);
  mark(0, s);
  cudaError_t e = launch_simt_rowproj(G, dtype, B, T, p, S, dtype, false, ir, W, s);
  if (e == cudaSuccess) e = launch_simt_colproj(A, dtype, B, T, d, W, ir, Z, s);
  mark(1, s);
  if (e == cudaSuccess) e = launch_simt_rowproj(A, dtype, B, T, d, Z, DPRC_F32, true, ir, W, s);
  if (e == cudaSuccess) e = launch_simt_colproj(G, dtype, B, T, p, W, ir, M, s);
  mark(2, s);
  if (e == cudaSuccess)
    e = launch_qr_project(M, B, p, ir, P, dtype, reinterpret_cast<float*>(w + sp.qscratch_off),
                          QP, false, s);
  mark(3, s);
  if (e == cudaSuccess)
    e = launch_simt_rowproj(G, dtype, B, T, p, QP, DPRC_F32, true, 2 * ir, W, s);
  if (e == cudaSuccess) e = launch_simt_colproj(A, dtype, B, T, d, W, 2 * ir, Y, s);
  if (e == cudaSuccess)
    e = launch_simt_norm_finish(Y, B, d, 2 * ir, ir, 1.0f / static_cast<float>(r), n, accumulate,
                                s);
  mark(4, s);
  return cuda_status(e);
}

dprc_status dprc_exact_norm_form(const void* A, const void* G, dprc_dtype dtype, int64_t B,
                                 int64_t T, int64_t d, int64_t p, int form, float* n,
                                 int accumulate, void* ws, size_t ws_bytes, void* stream) {
  DPRC_NVTX_RANGE();
  if (!A || !G || !n) return DPRC_ERR_NULL;
  dprc_status st = check_common(dtype, B, T, d, p);
  if (st != DPRC_OK) return st;
  if (!aligned16(A) || !aligned16(G) || !aligned16(n)) return DPRC_ERR_ALIGN;
  if (!ws) return DPRC_ERR_WORKSPACE;
  if (!aligned16(ws)) return DPRC_ERR_ALIGN;
  if (plan_exact(dtype, B, T, d, p, form).kind == ExactPlan::kNone) return DPRC_ERR_SHAPE;
  if (ws_bytes < plan_exact_bytes(dtype, B, T, d, p)) return DPRC_ERR_WORKSPACE;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  const ExactPlan e = plan_exact(dtype, B, T, d, p, form);  // with this device's SM count
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  mark(0, s);
  float* partials = reinterpret_cast<float*>(static_cast<char*>(ws) + exact_partials_off(B));
  cudaError_t err = cudaSuccess;
  switch (e.kind) {
    case ExactPlan::kDirectTc:
      err = launch_tc_exact_direct(A, G, B, T, d, p, partials, n, accumulate, s);
      break;
    case ExactPlan::kGhostTc:
      // the work queue's counters sit at the front of the zeroed counter block
      err = launch_tc_exact_ghost(A, G, B, T, d, p, e.W, ws, partials, n, accumulate, s);
      break;
    case ExactPlan::kNarrowTc:
      // per-sample tickets at the front of the zeroed counter block
      err = launch_narrow_norm(A, G, B, T, d, p, static_cast<int*>(ws), partials, n, accumulate,
                               s);
      break;
    default:
      err = launch_exact_ghost(A, G, dtype, B, T, d, p, partials, n, accumulate, s);
  }
  mark(1, s);
  return cuda_status(err);
}

dprc_status dprc_exact_norm(const void* A, const void* G, dprc_dtype dtype, int64_t B, int64_t T,
                            int64_t d, int64_t p, float* n, int accumulate, void* ws,
                            size_t ws_bytes, void* stream) {
  return dprc_exact_norm_form(A, G, dtype, B, T, d, p, DPRC_EXACT_AUTO, n, accumulate, ws,
                              ws_bytes, stream);
}

int dprc_exact_norm_plan(dprc_dtype dtype, int64_t B, int64_t T, int64_t d, int64_t p,
                         int form) {
  if (check_common(dtype, B, T, d, p) != DPRC_OK) return 0;
  if (!device_ok()) return 0;
  const ExactPlan e = plan_exact(dtype, B, T, d, p, form);
  switch (e.kind) {
    case ExactPlan::kDirectTc:
    case ExactPlan::kNarrowTc: return DPRC_EXACT_DIRECT;
    case ExactPlan::kGhostTc: return e.W == 1 ? DPRC_EXACT_GHOST_N128 : DPRC_EXACT_GHOST_N256;
    case ExactPlan::kGhostSimt: return DPRC_EXACT_GHOST;
    default: return 0;
  }
}

dprc_status dprc_clip_factors(const float* n, int64_t B, float C, float* c, int32_t* nonfinite,
                              void* stream) {
  DPRC_NVTX_RANGE();
  if (!n || !c) return DPRC_ERR_NULL;
  if (B < 1 || B > (int64_t(1) << 31)) return DPRC_ERR_SHAPE;
  if (!(C > 0.f) || !(C < __builtin_inff())) return DPRC_ERR_SHAPE;
  if (!aligned16(n) || !aligned16(c)) return DPRC_ERR_ALIGN;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  return cuda_status(launch_clip(n, B, C, c, nonfinite, static_cast<cudaStream_t>(stream)));
}

dprc_status dprc_add_noise(float* grad, int64_t N, float sigma, float C, uint64_t seed,
                           uint64_t step, void* stream) {
  DPRC_NVTX_RANGE();
  if (N < 0) return DPRC_ERR_SHAPE;
  if (N > 0 && !grad) return DPRC_ERR_NULL;
  if (!(sigma >= 0.f) || !(sigma < __builtin_inff()) || !(C >= 0.f) || !(C < __builtin_inff()))
    return DPRC_ERR_SHAPE;
  if (N > 0 && !aligned16(grad)) return DPRC_ERR_ALIGN;
  if (N == 0) return DPRC_OK;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  mark(0, s);
  const cudaError_t e = launch_noise(grad, N, sigma, C, seed, step, s);
  mark(1, s);
  return cuda_status(e);
}

dprc_status dprc_add_noise_at(void* grad, dprc_dtype dtype, int64_t N, uint64_t first_element,
                             float sigma, float C, uint64_t seed, uint64_t step, void* stream) {
  DPRC_NVTX_RANGE();
  if (dtype != DPRC_F32 && dtype != DPRC_BF16) return DPRC_ERR_DTYPE;
  if (N < 0) return DPRC_ERR_SHAPE;
  if (N > 0 && !grad) return DPRC_ERR_NULL;
  if (!(sigma >= 0.f) || !(sigma < __builtin_inff()) || !(C >= 0.f) || !(C < __builtin_inff()))
    return DPRC_ERR_SHAPE;
  // the stream has 2^66 elements; the call's range must not wrap
  if (static_cast<uint64_t>(N) > ~uint64_t(0) - first_element) return DPRC_ERR_SHAPE;
  if (N > 0 && !aligned16(grad)) return DPRC_ERR_ALIGN;
  if (N == 0) return DPRC_OK;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  mark(0, s);
  const cudaError_t e = launch_noise_at(grad, dtype, N, first_element, sigma, C, seed, step, s);
  mark(1, s);
  return cuda_status(e);
}

dprc_status dprc_philox_words(uint32_t* out, int64_t n_blocks, uint64_t first_block,
                              uint64_t seed, uint64_t step, void* stream) {
  DPRC_NVTX_RANGE();
  if (n_blocks < 0) return DPRC_ERR_SHAPE;
  if (n_blocks > 0 && !out) return DPRC_ERR_NULL;
  if (n_blocks > 0 && !aligned16(out)) return DPRC_ERR_ALIGN;
  if (n_blocks == 0) return DPRC_OK;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  return cuda_status(launch_philox_words(out, n_blocks, first_block, seed, step,
                                         static_cast<cudaStream_t>(stream)));
}

dprc_status dprc_test_hutch_fault(int mode, uint64_t wait_ns, int64_t L, const void* const* A,
                                  const void* const* G, const void* const* P, const int64_t* d,
                                  const int64_t* p, int64_t B, int64_t T, int64_t k, float* n,
                                  void* ws, size_t ws_bytes, void* stream) {
  DPRC_NVTX_RANGE();
  if (!A || !G || !P || !d || !p || !n) return DPRC_ERR_NULL;
  if (mode != kFaultReadyNeverMet && mode != kFaultClusterShape) return DPRC_ERR_SHAPE;
  constexpr uint64_t kMaxWaitNs = 2000000000ull;  // the kernels' own limit
  if (wait_ns < 1000 || wait_ns > kMaxWaitNs) return DPRC_ERR_SHAPE;
  if (L < 1 || L > kMaxFusedLayers) return DPRC_ERR_SHAPE;
  if (!fused_hutch_supported(k)) return DPRC_ERR_SHAPE;
  int64_t dmax = 0, pmax = 0;
  for (int64_t l = 0; l < L; ++l) {
    if (!A[l] || !G[l] || !P[l]) return DPRC_ERR_NULL;
    const dprc_status st = check_common(DPRC_BF16, B, T, d[l], p[l]);
    if (st != DPRC_OK) return st;
    if (!tc_path_supported(DPRC_BF16, B, T, d[l], p[l], k, false)) return DPRC_ERR_SHAPE;
    if (!aligned16(A[l]) || !aligned16(G[l]) || !aligned16(P[l])) return DPRC_ERR_ALIGN;
    dmax = std::max(dmax, d[l]);
    pmax = std::max(pmax, p[l]);
  }
  if (!aligned16(n)) return DPRC_ERR_ALIGN;
  if (!ws) return DPRC_ERR_WORKSPACE;
  if (!aligned16(ws)) return DPRC_ERR_ALIGN;
  const int layers = L > 1 ? kMaxFusedLayers : 1;
  const TcPlan t = plan_tc(DPRC_OP_HUTCH, B, T, dmax, pmax, k, layers);
  if (ws_bytes < t.total) return DPRC_ERR_WORKSPACE;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  HutchFaultTest test;
  test.mode = mode;
  test.wait_ns = wait_ns;
  bool launched = false;
  const cudaError_t e =
      launch_tc_hutch_fault_test(static_cast<int>(L), A, G, P, d, p, B, T, k,
                                 fused_scratch(t, static_cast<char*>(ws)), n, test,
                                 static_cast<cudaStream_t>(stream), &launched);
  if (!launched) {
    if (e != cudaSuccess) (void)cudaGetLastError();
    return e == cudaSuccess ? DPRC_ERR_SHAPE : DPRC_ERR_CUDA;
  }
  return cuda_status(e);
}

dprc_status dprc_device_error(int32_t* out, int reset) {
  if (!out) return DPRC_ERR_NULL;
  if (!device_ok()) return DPRC_ERR_DEVICE;
  cudaError_t (*const readers[])(int32_t*, bool) = {read_device_error_proj,
                                                     read_device_error_hutch,
                                                     read_device_error_exact,
                                                     read_device_error_qr,
                                                     read_device_error_narrow};
  int32_t first = 0;
  for (auto rd : readers) {
    int32_t v = 0;
    const cudaError_t e = rd(&v, reset != 0);
    if (e != cudaSuccess) return cuda_status(e);
    if (first == 0) first = v;
  }
  *out = first;
  return DPRC_OK;
}

}  // extern "C"
