// Host-side declarations shared by the libdprc translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dprc.h"

#include <nvtx3/nvToolsExt.h>

namespace dprc {

// One NVTX range per C-ABI call, named after the call, so the kernels of a
// call group under its name in a profiler's timeline (ncu --nvtx).  With no
// tool attached a push or pop is a check of an unset function pointer.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};
#define DPRC_NVTX_RANGE() ::dprc::NvtxRange dprc_nvtx_range_(__func__)


// ---- block schedules --------------------------------------------------------
// How one tensor-core launch assigns its blocks (128 output rows, `upb` units
// each) to CTAs: whole blocks, `bpc` per CTA (cl == 1), or one block per
// cluster of `cl` CTAs that split its units and reduce through distributed
// shared memory.
struct BlockSched {
  int cl = 1;
  int bpc = 1;
  int64_t nblocks = 0;
  int upb = 0;
  int grid = 0;
};
BlockSched make_block_sched(int64_t nblocks, int upb, int slots);

// Scratch layout of the tensor-core path of one Hutchinson or Hutch++ call.
// Most layers one fused Hutchinson launch takes (the per-layer tensor maps
// travel in the kernel parameters); calls with more layers use several
// launches.
constexpr int kMaxFusedLayers = 56;

struct TcPlan {
  int64_t tpad = 0;           // row stride (elements) of the [B][2n][tpad] sketches
  // counter block (zero between calls), the same for every plan:
  size_t stick_off = 0;       // tickets int32 [kMaxFusedLayers][B] (row 0: per-sample tickets)
  size_t ready_off = 0;       // sketch-ready counters int32 [kMaxFusedLayers][B]
  size_t lticket_off = 0;     // layers finished per sample int32 [B]
  size_t done2_off = 0;       // projection blocks finished per layer int32 [kMaxFusedLayers]
  size_t exit_off = 0;        // CTAs finished int32 [1]
  // scratch:
  size_t cnorm_off = 0;       // per-block squared norms fp32 [layers][B][chunks]
  size_t nl_off = 0;          // per-layer norms fp32 [layers][B]
  size_t w_off = 0, w_bytes = 0;  // sketch G P (or G S, A Z, G [Q|P']) hi/lo bf16
  size_t w2_off = 0;          // second and third sketch buffers (multi-layer calls; = w_off
  size_t w3_off = 0;          // otherwise)
  size_t z_off = 0;           // Hutch++: Z hi/lo bf16 [B][d][2r]
  size_t m_off = 0;           // Hutch++: M = O S fp32 [B][p][r]
  size_t qp_off = 0;          // Hutch++: [Q | P'] hi/lo bf16 [B][p][4r]
  size_t qscratch_off = 0;    // Hutch++: QR work space fp32 [B][p][r] * 2
  // Hutch++ with the QR beside the third pass (r = 16, cluster QR):
  size_t sp_off = 0;          // [S | P] bf16 [p][2r]
  size_t yp_off = 0;          // X P fp32 [B][d][r]
  size_t rc_off = 0;          // QR factors fp32 [B][qr_factor_floats()]
  size_t total = 0;
};

// Scratch layout of the SIMT (CUDA-core, fp32) path.
struct SimtPlan {
  size_t w_off = 0;   // [B][T][n] fp32 sketch
  size_t y_off = 0;   // [B][c][n] fp32 projection
  size_t z_off = 0;   // Hutch++ Z / M / [Q|P'] buffers
  size_t m_off = 0;
  size_t qp_off = 0;
  size_t qscratch_off = 0;
  size_t total = 0;
};

int device_sm_count();
// Argument checks of dprc_norm_hutch that need no device (pointers, sizes,
// alignment); DPRC_OK or the status the call returns.
dprc_status check_hutch_args(const void* A, const void* G, const void* P, dprc_dtype dtype,
                             int64_t B, int64_t T, int64_t d, int64_t p, int64_t k,
                             const float* n);
// Whether the current device is an sm_103 GPU (cached per device).
bool current_device_supported();
int rowproj_ctas_per_sm();
int colproj_ctas_per_sm(int nmma);
int colproj_stage_chunk();
int colproj_tile_t();
// Device error words of the translation units whose kernels wait (see
// common.cuh); dprc_device_error() reports the first nonzero one.
cudaError_t read_device_error_proj(int32_t* out, bool reset);
cudaError_t read_device_error_exact(int32_t* out, bool reset);
cudaError_t read_device_error_hutch(int32_t* out, bool reset);
cudaError_t read_device_error_qr(int32_t* out, bool reset);
bool tc_path_supported(dprc_dtype dt, int64_t B, int64_t T, int64_t d, int64_t p, int64_t k,
                       bool hutchpp);
BlockSched rowproj_sched(int64_t B, int64_t T, int64_t c, int nmma);
BlockSched colproj_sched(int64_t B, int64_t T, int64_t c, int nmma);

// Bytes of the counter block every workspace starts with (zero between calls).
size_t ctrl_bytes(int64_t B);
// `layers`: layer slots of the per-layer scratch (1 for single-layer calls,
// kMaxFusedLayers with two sketch buffers for dprc_norm_hutch_layers).
TcPlan plan_tc(dprc_op op, int64_t B, int64_t T, int64_t d, int64_t p, int64_t k,
               int layers = 1);
SimtPlan plan_simt(dprc_op op, int64_t B, int64_t T, int64_t d, int64_t p, int64_t k);
// Which kernel an exact-norm call runs (form: dprc_exact_form).
struct ExactPlan {
  enum Kind { kNone = 0, kDirectTc, kGhostTc, kGhostSimt, kNarrowTc };
  Kind kind = kNone;
  int W = 0;               // span width of the tensor-core ghost form
  int64_t per_sample = 0;  // partials per sample
};
ExactPlan plan_exact(dprc_dtype dt, int64_t B, int64_t T, int64_t d, int64_t p, int form);
size_t plan_exact_bytes(dprc_dtype dt, int64_t B, int64_t T, int64_t d, int64_t p);

// ---- tensor maps -----------------------------------------------------------
// 3-D bf16 tensor map over [dim2][dim1][dim0] (dim0 contiguous) with row
// strides in elements, a box of (box0, box1, 1) and the given swizzle bytes
// (0, 32, 64 or 128).
bool make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t dim0, uint64_t dim1,
                       uint64_t dim2, uint64_t stride1_elems, uint64_t stride2_elems,
                       uint32_t box0, uint32_t box1, int swizzle_bytes);

// ---- launchers (return cudaSuccess or the launch error) --------------------
// Row projection on tensor cores: W[i] = X[i] R[i] with X [B][T][c] bf16 and
// R [Rb][c][nmma] bf16 (Rb = 1: shared by the batch).  With hilo_in the two
// column halves of R are the hi and lo parts of one fp32 matrix and are
// summed.  W is written as bf16 hi/lo planes [B][2n][tpad].  CTA 0 also
// clears `zero_ints` int32 words at `zero_ptr` (the next kernel's tickets).
// beside_previous: a programmatic dependent launch that runs while the
// previous kernel in the stream (which must let it start early) still runs;
// X and R must not be written by that kernel.  CTA 0 waits for it before
// exiting, so this kernel completes after it.
// ready (may be null): int32 [B], zero on entry; every CTA adds one to
// ready[i] after each of its blocks of sample i is in memory (release), so a
// sample's count reaches ceil(T / 128) * bs.cl.
cudaError_t launch_tc_rowproj(const void* X, int64_t B, int64_t T, int64_t c, const void* R,
                              bool r_batched, int nmma, bool hilo_in, void* W, int64_t tpad,
                              const BlockSched& bs, int* zero_ptr, size_t zero_ints,
                              cudaStream_t s, bool beside_previous = false,
                              int* ready = nullptr);

// kColprojSplit: the first n_split = n / 2 columns of Y as bf16 hi/lo
// [B][c][n], the rest fp32 [B][c][n / 2]; kColprojF32Hilo: Y both ways;
// kColprojHpp (n = 16): Y = X M of Hutch++, whose head and tail
// ||Y_Q||^2 + ||Y_P - Y_Q C||^2 / 16 (Y_Q = Y diag(s) R^-1, hutchpp.cu) are
// added into n_out like kColprojNorm's squares, from the QR factors hpp_rc and
// Y_P = X P (fp32 [B][c][16]).
enum ColprojMode {
  kColprojNorm = 0,
  kColprojF32 = 1,
  kColprojHilo = 2,
  kColprojSplit = 3,
  kColprojF32Hilo = 4,
  kColprojHpp = 5
};

// Hutch++ combining step: a column j of R with |R_jj| at most this fraction of
// its column norm is left out of X Q (hutchpp.cu says why).
constexpr float kHppDropTau = 1e-3f;

// Column projection on tensor cores, reduced over T: Y[i] = X[i]^T W[i] with
// X [B][T][c] bf16 and W the hi/lo sketch [B][2n][tpad].  Mode kColprojNorm
// adds sum_j w_j ||Y[:, j]||^2 (w_j = 1 for j < n_head, w_tail otherwise) into
// n_out (per-block squares in chunk_norms, combined in block order by the
// last block of each sample, found with sample_tickets, which must be zero);
// kColprojF32 writes Y [B][c][n]; kColprojHilo writes Y as bf16 hi/lo [B][c][2n].
// ready (may be null): the counts of a launch_tc_rowproj with the same
// `ready` just before this one in the stream (pdl set): the loads of sample
// i's sketch wait for ready[i] >= ready_target instead of that kernel's end,
// so a sample's projection starts as soon as its sketch is written.  With
// ready_rows > 0 (kColprojNorm and kColprojHpp only) the sample's last block
// sets ready[r * B + i] back to zero for r < ready_rows, once every block is
// past its wait; counts of earlier launches may share that block of rows.
cudaError_t launch_tc_colproj(const void* X, int64_t B, int64_t T, int64_t c, const void* W,
                              int64_t tpad, int n, const BlockSched& bs, int* sample_tickets,
                              float* chunk_norms, ColprojMode mode, float* n_out, int accumulate,
                              int n_head, float w_tail, float* y_f32, void* y_hilo, bool pdl,
                              cudaStream_t s, int n_split = 0, const float* hpp_rc = nullptr,
                              const float* hpp_yp = nullptr, int* ready = nullptr,
                              int ready_target = 0, int ready_rows = 0);

// SIMT (fp32 CUDA-core) building blocks; Xdt is the dtype of X, Rdt of R.
cudaError_t launch_simt_rowproj(const void* X, dprc_dtype xdt, int64_t B, int64_t T, int64_t c,
                                const void* R, dprc_dtype rdt, bool r_batched, int n, float* W,
                                cudaStream_t s);
cudaError_t launch_simt_colproj(const void* X, dprc_dtype xdt, int64_t B, int64_t T, int64_t c,
                                const float* W, int n, float* Y, cudaStream_t s);
cudaError_t launch_simt_norm_finish(const float* Y, int64_t B, int64_t c, int n, int n_head,
                                    float w_tail, float* n_out, int accumulate, cudaStream_t s);

// Hutch++ middle step: per-sample Householder QR of M [B][p][r] (fp32),
// then P' = P - Q (Q^T P); writes [Q | P'] either as bf16 hi/lo [B][p][4r]
// (hilo = true) or fp32 [B][p][2r].  scratch: fp32 [B][p][r] * 2.
// Cluster QR (r = 16, 16 <= p <= 4096): one cluster of 8 CTAs per sample;
// same output as launch_qr_project.
bool qr_cluster_supported(int64_t p, int r);
// With rc set, also writes per sample (rc + i qr_factor_floats()) the R of the
// column-scaled M (16 x 16 row-major), the 16 column scales s (M diag(s) =
// Q R) and C = Q^T P (16 x 16); out may then be null (no [Q | P'] written).
// The launch lets the next kernel start at once (see launch_tc_rowproj).
cudaError_t launch_qr_cluster(const float* M, int64_t B, int64_t p, const void* P, dprc_dtype pdt,
                              void* out, bool hilo, cudaStream_t s, float* rc = nullptr);
int qr_factor_floats();

// Hutch++ with the QR beside the third pass (hutchpp.cu): SP = [S | P] row by
// row (bf16 [p][2r], r a multiple of 8), the first pass's sketch operand.
cudaError_t launch_pack_cols(const void* S, const void* P, void* SP, int64_t p, int r,
                             cudaStream_t s);
cudaError_t launch_qr_project(const float* M, int64_t B, int64_t p, int r, const void* P,
                              dprc_dtype pdt, float* scratch, void* out, bool hilo,
                              cudaStream_t s);

// Exact norm on tensor cores by the direct form: per sample, 128 x 256 tiles
// of A_i^T G_i accumulated over T in TMEM and squared in the epilogue; one
// partial per tile (fgc_partials(B, d, p) floats), summed per sample in index
// order into n_out.  bf16, d and p multiples of 8.
int64_t fgc_partials(int64_t B, int64_t d, int64_t p);
// Fused Hutchinson: sketch and projection of 1..kMaxFusedLayers layers as
// phases of one persistent launch (bf16, k = 16 or 32, one B and T for all
// layers).  n_out (+)= the layer sum.  Returns cudaSuccess with *launched
// false when the kernel cannot run with these shapes on this device (the
// caller then uses the two-kernel path); the counters must be zero and are
// zero again afterwards.
struct FusedScratch {
  void* W[3];           // sketch buffers (layer l uses W[l % 3]); all equal for one layer
  int64_t tpad;
  int* ready;           // [kMaxFusedLayers][B]
  int* tickets;         // [kMaxFusedLayers][B]
  int* lticket;         // [B]
  int* done2;           // [kMaxFusedLayers]
  int* exit_count;      // [1]
  float* chunk_norms;   // [layers][B][chunks]
  float* nl;            // [layers][B]
};
FusedScratch fused_scratch(const TcPlan& t, char* ws);
// The first two passes of Hutch++ (r = 16) as one persistent launch of the
// fused kernel: pass 1 sketches G with SP = [S | P] and writes Z = A^T G S as
// bf16 hi/lo [B][d][32] and X P = A^T G P fp32 [B][d][16]; pass 2 sketches A
// with Z_i as soon as all of Z_i is written and writes M = G^T A Z fp32
// [B][p][16] and hi/lo [B][p][32].  *launched is false when the shapes do not
// fit its plan (the caller then runs the passes as separate kernels).
cudaError_t launch_tc_hutchpp12(const void* A, const void* G, const void* SP, int64_t B,
                                int64_t T, int64_t d, int64_t p, const FusedScratch& ws, void* Z,
                                float* YP, float* M, void* MH, cudaStream_t s, bool* launched);

bool fused_hutch_supported(int64_t k);
// Whether a dprc_norm_hutch call with these sizes takes the fused kernel on
// the current device (the same decision the launcher makes).
bool fused_hutch_planned(int64_t B, int64_t T, int64_t d, int64_t p, int64_t k);
// Whether launch_tc_hutchpp12 would launch for these sizes on the current device.
bool hutchpp12_planned(int64_t B, int64_t T, int64_t d, int64_t p);
// Optional clip epilogue: c[i] = min(1, C / sqrt(n_out[i])) (the rule of
// dprc_clip_factors) once n_out[i] is final.
struct ClipOut {
  float C = 0.f;
  float* c = nullptr;
  int32_t* nonfinite = nullptr;
};
cudaError_t launch_tc_hutch_layers(int L, const void* const* A, const void* const* G,
                                   const void* const* P, const int64_t* d, const int64_t* p,
                                   int64_t B, int64_t T, int64_t k, const FusedScratch& ws,
                                   float* n_out, int accumulate, cudaStream_t s, bool* launched,
                                   const ClipOut* clip = nullptr);
// Failure-detection test of the fused kernel (dprc_test_hutch_fault): mode
// kFaultReadyNeverMet plans the launch as usual but raises every sketch-ready
// target by one, so the projection's waits cannot succeed; mode
// kFaultClusterShape launches a plan without clusters as clusters of 2.  Every
// wait in the launch is limited to wait_ns.  *launched false: these layers do
// not take the fused kernel (or, for the second mode, their plan has clusters).
enum { kFaultReadyNeverMet = 0, kFaultClusterShape = 1 };
struct HutchFaultTest {
  int mode = kFaultReadyNeverMet;
  unsigned long long wait_ns = 0;
};
cudaError_t launch_tc_hutch_fault_test(int L, const void* const* A, const void* const* G,
                                       const void* const* P, const int64_t* d, const int64_t* p,
                                       int64_t B, int64_t T, int64_t k, const FusedScratch& ws,
                                       float* n_out, const HutchFaultTest& test, cudaStream_t s,
                                       bool* launched);
// The +-1 projection variant on the fused kernel (bf16, k = 16 or 32, one
// layer): the signs are generated in the kernel from (seed, step); the norm is
// scaled by 1/k.  *launched false: not possible here (use the signs below).
cudaError_t launch_tc_hutch_pm1(const void* A, const void* G, int64_t B, int64_t T, int64_t d,
                                int64_t p, int64_t k, uint64_t seed, uint64_t step,
                                const FusedScratch& ws, float* n_out, int accumulate,
                                cudaStream_t s, bool* launched);
// S [p][k] in {-1, +1} (n = p k entries) written as dt, from the same stream.
cudaError_t launch_pm1_signs(void* out, dprc_dtype dt, int64_t n, uint64_t seed, uint64_t step,
                             cudaStream_t s);
cudaError_t launch_tc_exact_direct(const void* A, const void* G, int64_t B, int64_t T, int64_t d,
                                   int64_t p, float* partials, float* n_out, int accumulate,
                                   cudaStream_t s);
// Exact norm on tensor cores by the ghost form: per sample, 128-token row
// blocks against spans of W = 1 or 2 column blocks (upper triangle), the Gram
// tiles of A and of G in TMEM and their weighted dot product in the epilogue;
// one partial per unit (ghost_partials(B, T, W) floats), summed per sample in
// index order into n_out.  bf16, d and p multiples of 8.  `counters`: 16
// bytes, 8-byte aligned, zero on entry and left zero (the work queue).
int64_t ghost_partials(int64_t B, int64_t T, int W);
cudaError_t launch_tc_exact_ghost(const void* A, const void* G, int64_t B, int64_t T, int64_t d,
                                  int64_t p, int W, void* counters, float* partials,
                                  float* n_out, int accumulate, cudaStream_t s);
// Narrow layers (bf16, d and p multiples of 8, min(d, p) <= 64): the gradient
// X_i = A_i^T G_i formed tile by tile in one streaming tensor-core pass.
// launch_narrow_norm: n_out (+)= ||X_i||^2 (narrow_partials(B, d, p) floats
// of scratch); launch_narrow_hutch (narrow_proj_supported): n_out (+)=
// scale ||X_i P||^2 with P [p][k] bf16, or with the +-1 signs of (seed, step)
// when P is null (narrow_hutch_scratch_bytes of scratch).
bool narrow_supported(dprc_dtype dt, int64_t d, int64_t p);
bool narrow_proj_supported(dprc_dtype dt, int64_t d, int64_t p, int64_t k);
int64_t narrow_partials(int64_t B, int64_t d, int64_t p);
size_t narrow_hutch_scratch_bytes(int64_t B, int64_t d, int64_t p, int64_t k);
cudaError_t read_device_error_narrow(int32_t* out, bool reset);
// tickets: int32 [B], zero on entry and zero again on exit (one launch).
cudaError_t launch_narrow_norm(const void* A, const void* G, int64_t B, int64_t T, int64_t d,
                               int64_t p, int* tickets, float* partials, float* n_out,
                               int accumulate, cudaStream_t s);
// clip: the clip factors of the final n_out, written in the same launch
cudaError_t launch_narrow_hutch(const void* A, const void* G, const void* P, int64_t B,
                                int64_t T, int64_t d, int64_t p, int64_t k, float scale,
                                uint64_t seed, uint64_t step, int* tickets, float* partials,
                                float* n_out, int accumulate, cudaStream_t s,
                                const ClipOut* clip = nullptr);
// n_out[i] (+)= sum of partials[i * per_sample .. (i + 1) * per_sample), fixed order.
cudaError_t launch_partials_finish(const float* partials, int64_t B, int64_t per_sample,
                                   float* n_out, int accumulate, cudaStream_t s);
// Exact norm by the ghost form on CUDA cores (fp32 arithmetic, any layout),
// deterministic.
cudaError_t launch_exact_ghost(const void* A, const void* G, dprc_dtype dt, int64_t B,
                               int64_t T, int64_t d, int64_t p, float* partials, float* n_out,
                               int accumulate, cudaStream_t s);

cudaError_t launch_clip(const float* n, int64_t B, float C, float* c, int32_t* nonfinite,
                        cudaStream_t s);
cudaError_t launch_noise(float* grad, int64_t N, float sigma, float C, uint64_t seed,
                         uint64_t step, cudaStream_t s);
// grad[i] += sigma C z_{first_element + i}, grad fp32 or bf16 (sum in fp32,
// rounded once).
cudaError_t launch_noise_at(void* grad, dprc_dtype dt, int64_t N, uint64_t first_element,
                            float sigma, float C, uint64_t seed, uint64_t step, cudaStream_t s);
cudaError_t launch_philox_words(uint32_t* out, int64_t n_blocks, uint64_t first_block,
                                uint64_t seed, uint64_t step, cudaStream_t s);

}  // namespace dprc
