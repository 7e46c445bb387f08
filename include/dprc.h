/*
 * dprc.h - C ABI of libdprc, the GB300 (sm_103a) hot path of DP-SGD with
 * randomized clipping (DP-SGD-RC): per-sample, per-layer gradient-norm
 * estimation, clip factors and the Gaussian noise add.
 *
 * Source of the method: "Efficient DP-SGD for LLMs with Randomized Clipping"
 * (ICML 2026, arXiv 2605.24879), as described by the papernotes.org notes
 * ("Method > Overall framework", "Method > Key design") and the gist.science
 * technical summary ("Methodologie > Kernmechanisme", "Algorithmische Flow").
 *
 * Setting.  For one linear-like layer a forward hook captures the activations
 * A (B x T x d) and a backward hook the output gradients G (B x T x p).  The
 * per-sample weight gradient is A_i^T G_i, and its squared Frobenius norm is
 *     n_i = ||A_i^T G_i||_F^2 = trace(G_i^T A_i A_i^T G_i) = trace(O_i).
 * The norm-estimation routine returns an estimate n_hat_i^(l) per layer l; the
 * layerwise sum n_i = sum_l n_hat_i^(l) sets the clip factor min(1, C/sqrt(n_i))
 * that rescales sample i's loss; after the second backward pass the aggregated
 * gradient receives sigma*C*N(0, I) noise.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Pointers named as device pointers must point to device memory (or
 *    managed memory) that stays valid until the enqueued work completes.  The
 *    library never allocates or frees memory.  Scratch memory is passed in as
 *    `ws` (see dprc_workspace_bytes).  Zero a workspace once before its first
 *    use (e.g. cudaMemsetAsync): it starts with a block of per-sample
 *    counters that must read zero when a call begins.  Every call that ends
 *    without a device error (dprc_device_error) leaves that block zero again.
 *    The block has one size for every B <= 256, so one workspace serves any
 *    sequence of calls with B <= 256 and sizes that fit it.  Above 256 samples
 *    the block grows with B: zero the workspace again before a call with
 *    B > 256 unless the previous call on it had the same B.  After a device
 *    error, zero it again.  The rest of its contents are scratch.
 *  - `stream` is a cudaStream_t passed as void*; NULL means the legacy default
 *    stream.  Calls only enqueue work and return; results are ready when the
 *    stream reaches them.  Calls on different streams may run concurrently
 *    only if they use different workspaces and outputs.
 *  - Layouts are dense and row-major: A [B][T][d], G [B][T][p], P and S
 *    [p][k] (k contiguous), outputs [B].  Element types are given by `dtype`
 *    (DPRC_F32 = float32, DPRC_BF16 = bfloat16); A, G, P and S share it.
 *  - Argument errors (null pointers, non-positive or inconsistent sizes,
 *    misaligned pointers, a workspace that is too small) return an error code
 *    before anything is enqueued.  A failed kernel launch returns
 *    DPRC_ERR_CUDA.  Nothing throws across this boundary.
 *  - Every wait inside a kernel is bounded; a wait that runs out sets the
 *    device error word that dprc_device_error() reads, and the kernel returns.
 *  - `accumulate` = 0 overwrites n[i]; `accumulate` != 0 adds to it, which is
 *    how the layerwise sum is formed across layers.
 */
#ifndef DPRC_H
#define DPRC_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DPRC_ABI_VERSION 1


typedef enum {
    DPRC_OK = 0,
    DPRC_ERR_NULL = 1,        /* a required pointer is NULL */
    DPRC_ERR_SHAPE = 2,       /* a size is out of range or inconsistent */
    DPRC_ERR_DTYPE = 3,       /* unknown dtype */
    DPRC_ERR_ALIGN = 4,       /* a pointer is not 16-byte aligned */
    DPRC_ERR_WORKSPACE = 5,   /* ws_bytes < dprc_workspace_bytes(...) or ws NULL */
    DPRC_ERR_CUDA = 6,        /* a CUDA runtime/driver call failed */
    DPRC_ERR_NONFINITE = 7,   /* reserved: reported through counters, not returns */
    DPRC_ERR_DEVICE = 8,      /* no usable sm_103 device for this call */
    DPRC_ERR_TOO_LARGE = 9    /* needs more scratch than the built-in buffer holds */
} dprc_status;

typedef enum { DPRC_F32 = 0, DPRC_BF16 = 1 } dprc_dtype;

typedef enum {
    DPRC_OP_HUTCH = 1,
    DPRC_OP_HUTCHPP = 2,
    DPRC_OP_EXACT = 3,
    DPRC_OP_HUTCH_LAYERS = 4,
    DPRC_OP_HUTCH_PM1 = 5,
    DPRC_OP_HUTCH_HOST = 6   /* the stage buffer of dprc_norm_hutch_clip_host */
} dprc_op;

/* Version of this ABI (DPRC_ABI_VERSION of the built library). */
int dprc_abi_version(void);

/* Short static description of a status code. */
const char* dprc_status_string(dprc_status s);

/*
 * Scratch bytes needed by one call of `op` with these sizes.  k is the
 * projection width for DPRC_OP_HUTCH, DPRC_OP_HUTCH_PM1 and
 * DPRC_OP_HUTCH_HOST, the sketch width r for DPRC_OP_HUTCHPP, and ignored
 * for DPRC_OP_EXACT.  For DPRC_OP_HUTCH_LAYERS, d and p are the largest
 * widths of the layer list.  DPRC_OP_HUTCH_HOST gives the size of the device
 * stage buffer of dprc_norm_hutch_clip_host.  Returns 0 for invalid sizes.
 * The size depends on the current device's SM count.
 */
size_t dprc_workspace_bytes(dprc_op op, dprc_dtype dtype, int64_t B, int64_t T,
                            int64_t d, int64_t p, int64_t k);

/*
 * Hutchinson estimate of each sample's squared gradient norm for one layer:
 *     n_hat_i = trace(P^T O_i P) = ||A_i^T (G_i P)||_F^2.
 * (papernotes.org, "Key design > Hutchinson random projection": the sketch
 *  Y = A^T (G P) is formed without the d x p gradient or any T x T matrix.)
 *  A  device [B][T][d], G device [B][T][p], P device [p][k], all `dtype`.
 *     P is one projection shared by the batch, entries N(0, 1/k) drawn by the
 *     caller (a fresh P per layer and step).
 *  n  device float [B]: n[i] = (accumulate ? n[i] : 0) + n_hat_i.
 *  Sizes: B >= 1, T >= 1, d >= 1, p >= 1, 1 <= k <= 256.
 *  Arithmetic: products and sums in fp32 (bf16 inputs are exact in fp32).
 *  For bf16 layers with one width <= 64 (adapter maps: p <= 64, or d <= 32
 *  with k <= 128) the small gradient X_i = A_i^T G_i is formed tile by tile in
 *  one pass and n_hat_i = ||X_i P||_F^2, the same quantity up to rounding.
 *  All pointers 16-byte aligned.  The result is deterministic for fixed
 *  inputs, sizes and device.
 */
dprc_status dprc_norm_hutch(const void* A, const void* G, const void* P, dprc_dtype dtype,
                            int64_t B, int64_t T, int64_t d, int64_t p, int64_t k,
                            float* n, int accumulate, void* ws, size_t ws_bytes, void* stream);

/*
 * dprc_norm_hutch followed by the clip factors of the updated n (the next
 * step of the method, papernotes.org, "Method > Overall framework"):
 *     n[i] (+)= || A_i^T (G_i P) ||_F^2,   c[i] = min(1, C / sqrt(n[i]))
 * with the rule of dprc_clip_factors (n = 0 gives 1; a non-finite or
 * negative n gives 0 and is counted in *nonfinite, which may be NULL).  Use
 * it for the last layer of a step.  When dprc_norm_hutch_launches reports one
 * launch, the clip factors are written by that launch's per-sample finishing
 * step (no second kernel); otherwise the clip kernel follows on the same
 * stream.  The results equal dprc_norm_hutch then dprc_clip_factors bit for
 * bit.
 *  c device float [B], 16-byte aligned; C > 0 and finite.  Other arguments,
 *  the workspace and errors as dprc_norm_hutch.
 */
dprc_status dprc_norm_hutch_clip(const void* A, const void* G, const void* P, dprc_dtype dtype,
                                 int64_t B, int64_t T, int64_t d, int64_t p, int64_t k,
                                 float* n, int accumulate, float C, float* c,
                                 int32_t* nonfinite, void* ws, size_t ws_bytes, void* stream);

/*
 * dprc_norm_hutch_clip (accumulate = 0) for inputs that are in HOST memory,
 * with the results written back to host memory: the whole per-sample norm and
 * clip step of one layer, from the host's tensors to the host's clip factors.
 *     n[i] = || A_i^T (G_i P) ||_F^2,   c[i] = min(1, C / sqrt(n[i]))
 *  A host [B][T][d], G host [B][T][p], P host [p][k], all `dtype`; n, c host
 *  float [B]; n may be NULL (the norms are then not copied back).  Use
 *  page-locked (pinned) host memory: the copies are then asynchronous and run
 *  at the host link's rate; pageable memory works, but its copies block the
 *  calling thread.
 *  The samples go to the device in chunks (the fewest samples that make at
 *  least 128 MB of A and G) on two internal copy streams (A and G side by
 *  side), through two slots of the stage buffer; each chunk's norms and clip
 *  factors are computed on `stream` as soon as its copies have landed, while
 *  the next chunk is copied, so only the last chunk's kernels do not hide
 *  under a copy.  n and c are copied back at the end, on
 *  `stream`: they are valid once `stream` reaches that point (synchronise it
 *  before reading them).  The per-sample results equal dprc_norm_hutch_clip
 *  on the device copies of a chunk bit for bit.
 *  stage: device buffer of dprc_workspace_bytes(DPRC_OP_HUTCH_HOST, dtype, B,
 *  T, d, p, k) bytes, 16-byte aligned; zero it once before its first use (it
 *  holds workspaces, placed by the sizes).  Calls with the same sizes may reuse
 *  it as it is; zero it again before a call with other sizes.  One call at a
 *  time may use a stage buffer.
 *  C > 0 and finite.  Errors as dprc_norm_hutch; a failed copy returns
 *  DPRC_ERR_CUDA.  No counterpart on the pages (the host side of one step).
 */
dprc_status dprc_norm_hutch_clip_host(const void* A, const void* G, const void* P,
                                      dprc_dtype dtype, int64_t B, int64_t T, int64_t d,
                                      int64_t p, int64_t k, float C, float* n, float* c,
                                      void* stage, size_t stage_bytes, void* stream);

/*
 * Hutchinson estimate with a +-1 projection generated from a seed (the {-1, +1}
 * one-bit projection the notes name as the way to cut P's memory further;
 * papernotes.org, "Experiments > Ablation".  The pages give no formula and
 * say its privacy analysis would have to be redone):
 *     n[i] (+)= (1/k) || A_i^T (G_i S) ||_F^2,   S [p][k] in {-1, +1}
 *  Entry (u, v) of S is bit (e & 31) of word ((e >> 5) & 3) of block (e >> 7),
 *  e = u k + v, of the Philox4x32-10 stream of (seed, step) (the block layout
 *  of dprc_philox_words); bit 1 gives -1.  For bf16 with k = 16 or 32 the
 *  signs are generated inside the kernel and never stored; other shapes write
 *  S into the workspace first.  The 1/k scale is exact for powers of two.
 *  Workspace: dprc_workspace_bytes(DPRC_OP_HUTCH_PM1, ...).  Other arguments
 *  and errors as dprc_norm_hutch.
 */
dprc_status dprc_norm_hutch_pm1(const void* A, const void* G, uint64_t seed, uint64_t step,
                                dprc_dtype dtype, int64_t B, int64_t T, int64_t d, int64_t p,
                                int64_t k, float* n, int accumulate, void* ws, size_t ws_bytes,
                                void* stream);

/*
 * Layerwise sum of Hutchinson estimates over the L linear layers of a model
 * (papernotes.org, "Method > Overall framework": n_i = sum_l n_hat_i^(l)):
 *     n[i] (+)= sum_l || A_l,i^T (G_l,i P_l) ||_F^2
 *  A, G, P: host arrays of L device pointers, layer l holding A [B][T][d[l]],
 *  G [B][T][p[l]] and P [p[l]][k]; d, p: host arrays of L sizes.  B, T, k and
 *  dtype are shared by all layers.  The result equals L dprc_norm_hutch calls
 *  with accumulate set after the first, except that the layer sum is added in
 *  layer order after all layers (a fixed order: bitwise repeatable).  For bf16
 *  and k = 16 or 32 the layers run in one persistent launch per 56 layers, so
 *  one layer's start-up and tail overlap its neighbours' streaming; otherwise
 *  they run one call at a time.  Workspace: dprc_workspace_bytes(
 *  DPRC_OP_HUTCH_LAYERS, dtype, B, T, max_l d[l], max_l p[l], k).  Errors as
 *  dprc_norm_hutch (checked for every layer before anything is enqueued).
 */
dprc_status dprc_norm_hutch_layers(int64_t L, const void* const* A, const void* const* G,
                                   const void* const* P, const int64_t* d, const int64_t* p,
                                   dprc_dtype dtype, int64_t B, int64_t T, int64_t k, float* n,
                                   int accumulate, void* ws, size_t ws_bytes, void* stream);

/*
 * dprc_norm_hutch_layers followed by the clip factors of the layer sum:
 *     n[i] (+)= sum_l || A_l,i^T (G_l,i P_l) ||_F^2,   c[i] = min(1, C / sqrt(n[i]))
 * (papernotes.org, "Method > Overall framework": the layerwise sum sets the
 * clip factor), with the rule of dprc_clip_factors.  The launch that adds the
 * last layer writes c in its per-sample finishing step; calls that take the
 * layers one at a time end with the clip kernel.  Arguments, workspace and
 * errors as dprc_norm_hutch_layers, plus C, c and nonfinite as
 * dprc_norm_hutch_clip.
 */
dprc_status dprc_norm_hutch_layers_clip(int64_t L, const void* const* A, const void* const* G,
                                        const void* const* P, const int64_t* d, const int64_t* p,
                                        dprc_dtype dtype, int64_t B, int64_t T, int64_t k,
                                        float* n, int accumulate, float C, float* c,
                                        int32_t* nonfinite, void* ws, size_t ws_bytes,
                                        void* stream);

/*
 * Number of kernels one dprc_norm_hutch call with these arguments enqueues on
 * the current device: 1 (bf16, k = 16 or 32: sketch and projection as two
 * phases of one persistent launch; or the one-pass kernel of a narrow
 * layer), 2 (other tensor-core shapes: a sketch kernel and a projection
 * kernel) or 3 (the CUDA-core path: sketch, projection, reduction).  0 for
 * arguments dprc_norm_hutch would reject or when no sm_103 device is current.
 * Enqueues nothing; for launch accounting and graph builders.  No counterpart
 * on the pages (a library property).
 */
int dprc_norm_hutch_launches(dprc_dtype dtype, int64_t B, int64_t T, int64_t d, int64_t p,
                             int64_t k);

/*
 * Number of kernels one dprc_norm_hutchpp call with these arguments enqueues
 * on the current device: 5 (bf16, r = 16, p <= 4096 and sizes that fit the
 * fused kernel's plan: the pack of [S | P], passes 1 and 2 in one launch, the
 * cluster QR, the third pass's sketch and its projection), 8 (the same shapes
 * with passes 1 and 2 as four kernels; or the CUDA-core path: three sketch and
 * projection pairs, the QR and a reduction) or 7 (other tensor-core shapes:
 * three pairs and the QR between the second and the third).  0 for arguments
 * dprc_norm_hutchpp would reject or when no sm_103 device is current.
 * Enqueues nothing.  No counterpart on the pages (a library property).
 */
int dprc_norm_hutchpp_launches(dprc_dtype dtype, int64_t B, int64_t T, int64_t d, int64_t p,
                               int64_t r);

/*
 * Hutch++ head/tail estimate for one layer (papernotes.org, "Key design >
 * Hutch++ head-tail decomposition"; gist.science, "Kernmechanisme" item 2):
 *     Q_i     = orthonormal basis of Col(O_i S)          (p x r, thin QR)
 *     n_hat_i = ||A_i^T G_i Q_i||_F^2 + (1/r) ||A_i^T G_i (I - Q_i Q_i^T) P||_F^2
 *  S, P device [p][r], `dtype`, entries N(0, 1) drawn by the caller and shared
 *  by the batch.  O_i S is formed as G_i^T (A_i (A_i^T (G_i S))); the QR is a
 *  per-sample Householder QR in fp32.  Sizes as dprc_norm_hutch with
 *  1 <= r <= 64.  Other arguments as dprc_norm_hutch.
 *  For bf16 with r = 16 and p <= 4096 the call enqueues the pack of [S | P],
 *  three (sketch, projection) pairs (the first two in one launch where its
 *  plan fits, pass 2 of a sample starting once pass 1 has written it) and the
 *  QR, which runs beside the third sketch: that pass streams
 *  A_i^T G_i M_i (M_i = O_i S) and its epilogue
 *  forms A_i^T G_i Q_i = (A_i^T G_i M_i) diag(s) R^-1 from the QR of the
 *  column-scaled M_i, leaving out a column of R whose diagonal is at most
 *  1e-3 of its norm (M_i numerically rank deficient there; the estimate then
 *  uses the remaining columns for the head and the residual of those for the
 *  tail).  Otherwise the QR runs between the second and third passes and the
 *  third pass streams [Q_i | P - Q_i (Q_i^T P)].
 */
dprc_status dprc_norm_hutchpp(const void* A, const void* G, const void* S, const void* P,
                              dprc_dtype dtype, int64_t B, int64_t T, int64_t d, int64_t p,
                              int64_t r, float* n, int accumulate, void* ws, size_t ws_bytes,
                              void* stream);

/*
 * Exact squared norm n_i = ||A_i^T G_i||_F^2, the quantity the estimators
 * approximate (the comparison path the pages set the method against;
 * papernotes.org, "Research background" and "Key design"; the pages weigh the
 * full-gradient form, O(T d p) per sample, against ghost clipping,
 * O(T^2 (d + p))).  Two exact forms:
 *   - direct: the d x p product A_i^T G_i formed in 128 x 256 tiles in
 *     on-chip memory and squared there (never stored);
 *   - ghost:  n_i = sum_{t,s} (A_i A_i^T)_{ts} (G_i G_i^T)_{ts}, tile by tile
 *     over the upper triangle of 128-token blocks (no T x T matrix stored).
 * bf16 with d and p multiples of 8 runs both on tensor cores (the ghost form
 * up to T = 65536); other layouts run the ghost form on CUDA cores (fp32,
 * T <= 2097120).  dprc_exact_norm takes the form with less tensor work for
 * these sizes on the current device (ghost when T < 2 d p / (d + p) and the
 * batch has enough 128-token blocks to keep every SM busy);
 * dprc_exact_norm_form lets the caller choose.  Both sum in a fixed order
 * (bitwise repeatable for fixed inputs, sizes, form and device).  Both
 * accumulate in fp32; the ghost form adds T^2 signed products whose sum can
 * be much smaller than its terms, so its rounding error scales with
 * (sum_t ||A_i[t]|| ||G_i[t]||)^2 rather than with n_i (a sum that rounding
 * takes below zero is returned as 0).  Arguments as
 * dprc_norm_hutch without P and k; the workspace size comes from
 * dprc_workspace_bytes(DPRC_OP_EXACT, ...) and covers every form.
 */
dprc_status dprc_exact_norm(const void* A, const void* G, dprc_dtype dtype, int64_t B,
                            int64_t T, int64_t d, int64_t p, float* n, int accumulate,
                            void* ws, size_t ws_bytes, void* stream);

typedef enum {
    DPRC_EXACT_AUTO = 0,        /* the form dprc_exact_norm takes */
    DPRC_EXACT_DIRECT = 1,      /* A_i^T G_i; tensor-core layout only */
    DPRC_EXACT_GHOST = 2,       /* sum_{t,s} (A A^T)_{ts} (G G^T)_{ts} */
    DPRC_EXACT_GHOST_N128 = 3,  /* ghost, Gram tiles 128 x 128 (tensor cores) */
    DPRC_EXACT_GHOST_N256 = 4   /* ghost, Gram tiles 128 x 256 (tensor cores) */
} dprc_exact_form;

/*
 * dprc_exact_norm with the form chosen by the caller (a dprc_exact_form).
 * GHOST takes the tile width with less work for these sizes; GHOST_N128 and
 * GHOST_N256 fix it (tensor-core layout only).  DPRC_ERR_SHAPE for an unknown
 * form, for DIRECT or a fixed tile width outside the tensor-core layout and
 * for a ghost form beyond its T limit.  Other errors as dprc_exact_norm.
 */
dprc_status dprc_exact_norm_form(const void* A, const void* G, dprc_dtype dtype, int64_t B,
                                 int64_t T, int64_t d, int64_t p, int form, float* n,
                                 int accumulate, void* ws, size_t ws_bytes, void* stream);

/*
 * The form a dprc_exact_norm_form call with these arguments runs on the
 * current device: DPRC_EXACT_DIRECT, DPRC_EXACT_GHOST_N128 or
 * DPRC_EXACT_GHOST_N256 on tensor cores, DPRC_EXACT_GHOST on CUDA cores; 0
 * when it would be rejected or no sm_103 device is current.  Enqueues nothing.
 */
int dprc_exact_norm_plan(dprc_dtype dtype, int64_t B, int64_t T, int64_t d, int64_t p,
                         int form);

/*
 * Clip factors c_i = min(1, C / sqrt(n_i)) (papernotes.org, "Method > Overall
 * framework").  n_i = 0 gives 1.  A non-finite or negative n_i gives 0 and is
 * counted in *nonfinite (device int32, may be NULL; the count is added to it).
 *  n, c device float [B]; B >= 1; C > 0 and finite.
 */
dprc_status dprc_clip_factors(const float* n, int64_t B, float C, float* c,
                              int32_t* nonfinite, void* stream);

/*
 * Gaussian noise add on the aggregated gradient: grad[e] += sigma * C * z_e
 * (papernotes.org, "Method > Overall framework": the aggregated gradient plus
 * sigma*C*N(0, I)).  z_e comes from the Philox4x32-10 stream of
 * dprc_philox_words: word (e & 3) of block (e >> 2), Box-Muller on the word
 * pairs (w0, w1) and (w2, w3) with u1 = ((w_a >> 8) + 1) * 2^-24 and
 * u2 = (w_b >> 8) * 2^-24:  z_a = sqrt(-2 ln u1) cos(2 pi u2),
 * z_b = sqrt(-2 ln u1) sin(2 pi u2), evaluated in fp32 with the hardware
 * logarithm, sine and cosine (|error| <= 2e-6 + 1e-6 r, r = sqrt(z_a^2 + z_b^2));
 * the integer stream itself is exact.  Any 1/B averaging belongs to the caller.
 *  grad device float [N], in place, 16-byte aligned; N >= 0; sigma >= 0.
 *  The same (seed, step) gives the same noise on every call and device.
 */
dprc_status dprc_add_noise(float* grad, int64_t N, float sigma, float C, uint64_t seed,
                           uint64_t step, void* stream);

/*
 * dprc_add_noise on one piece of a gradient that the caller keeps in several
 * buffers (one per weight, say), without gathering them into one: the pieces
 * laid end to end form the aggregated gradient, and the piece that starts at
 * element first_element of it gets the same noise as that range would get
 * from dprc_add_noise on the whole (papernotes.org, "Method > Overall
 * framework": sigma*C*N(0, I) on the aggregated gradient):
 *     grad[i] += sigma * C * z_{first_element + i},   0 <= i < N
 * with z_e as in dprc_add_noise.  dtype DPRC_F32 or DPRC_BF16: a bf16
 * gradient gets its sum formed in fp32 and rounded once to nearest.
 *  grad device [N] of dtype, in place, 16-byte aligned; N >= 0;
 *  first_element + N must not exceed 2^64.  Errors as dprc_add_noise, plus
 *  DPRC_ERR_DTYPE.
 */
dprc_status dprc_add_noise_at(void* grad, dprc_dtype dtype, int64_t N, uint64_t first_element,
                              float sigma, float C, uint64_t seed, uint64_t step, void* stream);

/*
 * The raw Philox4x32-10 stream behind dprc_add_noise (Salmon et al.,
 * "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11): block j is the
 * generator applied to the counter (j_lo, j_hi, step_lo, step_hi) under the
 * key (seed_lo, seed_hi).  Writes blocks [first_block, first_block + n_blocks)
 * as out[4*(j - first_block) + w], w = 0..3.
 *  out device uint32 [4 * n_blocks], 16-byte aligned; n_blocks >= 0.
 */
dprc_status dprc_philox_words(uint32_t* out, int64_t n_blocks, uint64_t first_block,
                              uint64_t seed, uint64_t step, void* stream);

/*
 * Reads (and, if reset != 0, clears) the device error word of the current
 * device.  Nonzero means a bounded in-kernel wait ran out, or a kernel
 * refused a launch shape it was not planned for (the value encodes which: see
 * DPRC_DEVERR_*); the affected outputs are invalid, and the workspace of the
 * call must be zeroed again before its next use.  The first error since the
 * last reset is kept.  This call synchronizes with the device.
 */
#define DPRC_DEVERR_PIPE_FULL 1   /* consumer waited too long for a tile */
#define DPRC_DEVERR_PIPE_EMPTY 2  /* producer waited too long for a free stage */
#define DPRC_DEVERR_ACCUM 3       /* epilogue waited too long for the accumulator */
#define DPRC_DEVERR_CLUSTER 4     /* a CTA waited too long for its cluster peers' partials */
#define DPRC_DEVERR_READY 5       /* the projection waited too long for a sample's sketch */
#define DPRC_DEVERR_LAUNCH 6      /* a kernel found its launch's cluster shape other than
                                     planned and returned before doing anything */
#define DPRC_DEVERR_BOUNDS 7      /* bounds-checked build only (libdprc_debug.so): an index
                                     failed its check and the access was skipped; the
                                     word's bits above the low 8 hold the source line */
dprc_status dprc_device_error(int32_t* out, int reset);

/*
 * Failure-detection test of the one-launch Hutchinson kernel (a check of this
 * library's own promise that every wait inside a kernel is bounded; the pages
 * have no counterpart).  The layers are given as for dprc_norm_hutch_layers
 * (bf16, k = 16 or 32, 1 <= L <= 56, widths multiples of 8, none narrow); the
 * launch is planned exactly as dprc_norm_hutch_layers (L > 1) or
 * dprc_norm_hutch (L = 1) plans it, with accumulate = 0, and then altered:
 *   mode 0: every sketch-ready target is set one above what the sketch phase
 *           adds, so no projection block's wait for its sample's sketch can
 *           succeed.  Each such wait runs out after wait_ns, sets
 *           DPRC_DEVERR_READY, and the launch unwinds: the other roles of a
 *           CTA stop at their next wait, the MMAs and copies already issued
 *           complete, the tensor memory is freed and the kernel returns.  n
 *           is not written.  The workspace's counters are left nonzero: zero
 *           it before its next use.
 *   mode 1: a plan without clusters is launched with clusters of 2; the
 *           kernel finds the cluster shape it was not planned for, sets
 *           DPRC_DEVERR_LAUNCH and returns before touching any memory (n and
 *           the workspace are unchanged).
 *  wait_ns: limit of the launch's waits on other CTAs' progress, 1e3 .. 2e9
 *           ns (the default is 2e9); waits inside a CTA or its cluster get
 *           twice that, so the wait that is the cause runs out first.
 *  Workspace: dprc_workspace_bytes(L > 1 ? DPRC_OP_HUTCH_LAYERS :
 *  DPRC_OP_HUTCH, ...).  Returns DPRC_ERR_SHAPE when the layers do not take
 *  the one-launch kernel on this device, or (mode 1) when its plan already
 *  uses clusters.  Other errors as dprc_norm_hutch_layers.  Read the result
 *  with dprc_device_error(&v, 1).
 */
dprc_status dprc_test_hutch_fault(int mode, uint64_t wait_ns, int64_t L, const void* const* A,
                                  const void* const* G, const void* const* P, const int64_t* d,
                                  const int64_t* p, int64_t B, int64_t T, int64_t k, float* n,
                                  void* ws, size_t ws_bytes, void* stream);

/*
 * Timing hook.  With events != NULL, every later call made by this host
 * thread records events[0] on its stream before its first kernel and
 * events[s] after its s-th stage (up to n_events - 1 stages; a stage is one
 * or two kernels: dprc_norm_hutch has 2 - the sketch G P and the projection
 * with its norm; dprc_norm_hutchpp has 4 - Z, M, the QR step, the final pass).
 * `events` are cudaEvent_t passed as void*, owned by the caller and valid
 * while set.  Recording between kernels disables the overlap of dependent
 * launches, so time whole calls with this hook off.  events = NULL,
 * n_events = 0 turns it off.
 */
dprc_status dprc_set_phase_events(void** events, int n_events);

/*
 * dprc_norm_hutch without a workspace argument, for callers that cannot
 * allocate device memory where they need the norm: code inside a framework
 * that owns the device allocator and forbids direct cudaMalloc, loops where a
 * (possibly device-synchronizing) allocation is not acceptable, or hooks and
 * plugins that are handed only input and output pointers.  The method's
 * pages have no counterpart to this entry point.
 *
 * Scratch: a fixed array of DPRC_NOALLOC_SCRATCH_BYTES in the library's own
 * device memory (a file-scope __device__ array), held on every GPU that loads
 * the library until the process exits.  Calls whose dprc_workspace_bytes
 * (DPRC_OP_HUTCH, ...) exceeds that size return DPRC_ERR_TOO_LARGE before
 * any device work, as do argument errors (the checks and codes of
 * dprc_norm_hutch) and DPRC_ERR_DEVICE when the current device is not an
 * sm_103 GPU.  The call itself allocates nothing (no cudaMalloc, cudaFree or
 * allocating library routine).
 *
 * Set-up: the first call on each device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current and caches it, so make the
 * first call on a device before any stream capture.
 *
 * Sharing: every call on a device uses the same array, which keeps the last
 * call's contents.  Its leading counter block must read zero when a call
 * begins, so each call first clears it on `stream` (cudaMemsetAsync, which
 * allocates nothing); no stale state from an earlier call, even one that hit
 * a device error, carries over.  Calls that can overlap on the
 * GPU (different streams, or different host threads) race on the array: the
 * caller must order them.  Arguments and results otherwise as dprc_norm_hutch.
 */
#define DPRC_NOALLOC_SCRATCH_BYTES (48u << 20)
dprc_status dprc_norm_hutch_noalloc(const void* A, const void* G, const void* P,
                                    dprc_dtype dtype, int64_t B, int64_t T, int64_t d,
                                    int64_t p, int64_t k, float* n, int accumulate,
                                    void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DPRC_H */
