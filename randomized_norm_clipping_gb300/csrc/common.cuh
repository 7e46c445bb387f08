// Device helpers shared by the libdprc kernels: bounded mbarrier waits, TMA
// tile loads, tcgen05 (TMEM allocation, MMA, commit, loads) and the shared
// memory / instruction descriptors of the 5th-generation tensor cores.
// Everything here is written as inline PTX for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "dprc.h"

namespace dprc {

// ---------------------------------------------------------------------------
// Device error word.  A bounded wait that runs out records its code here
// (first writer wins) and the kernel unwinds.  Internal linkage: the word read
// by dprc_device_error() is the copy in the translation unit that holds the
// pipelined (waiting) kernels.
// ---------------------------------------------------------------------------
static __device__ int g_device_error = 0;

// Host side: reads (and with `reset` clears) this translation unit's copy of
// the error word.  Every unit whose kernels wait exposes one of these, and
// dprc_device_error() combines them.
static inline cudaError_t read_tu_device_error(int32_t* out, bool reset) {
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

// Upper bound on any single in-kernel wait (ns of %globaltimer).
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void record_error(int code) {
  atomicCAS(&g_device_error, 0, code);
}

// Bounds-checked build (DPRC_DEBUG, built as libdprc_debug.so): every
// computed global or distributed-shared-memory index is checked before its
// access with DPRC_IN(cond).  A failed check records DPRC_DEVERR_BOUNDS with
// the source line in the bits above the code (first writer wins) and the
// access is skipped: no trap, the context stays usable and the host reads
// where it happened.  Release builds compile the checks away.
#ifdef DPRC_DEBUG
__device__ __forceinline__ bool dbg_in(bool ok, int line) {
  if (!ok) atomicCAS(&g_device_error, 0, DPRC_DEVERR_BOUNDS | (line << 8));
  return ok;
}
#define DPRC_IN(cond) ::dprc::dbg_in(static_cast<bool>(cond), __LINE__)
#else
#define DPRC_IN(cond) true
#endif

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------------------
// mbarrier
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for the phase with the given parity to complete.  Returns false (and
// records `code`) if it has not completed within kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, int code) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    for (int spin = 0; spin < 64; ++spin)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      record_error(code);
      return false;
    }
  }
}

// Like mbar_wait, with the time limit given by the caller, and giving up
// early (false, nothing recorded: the CTA is already unwinding) once another
// role of the CTA has set `abort` (may be null).  For the pipeline waits of a
// kernel whose roles stop at the first failure of any of them.
__device__ __forceinline__ bool mbar_wait_lim(uint64_t* bar, uint32_t parity, int code,
                                              unsigned long long limit_ns,
                                              const volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    for (int spin = 0; spin < 64; ++spin)
      if (mbar_try_wait(bar, parity)) return true;
    if (abort != nullptr && *abort != 0) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      record_error(code);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// Counters in global memory written by other CTAs (a release add after the
// data it announces) and waited on with acquire loads.
// ---------------------------------------------------------------------------
__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Bounded wait until *p >= target (acquire); false on timeout (error
// recorded) or once the CTA's abort flag is set (nothing recorded).
__device__ __forceinline__ bool wait_geq(const int* p, int target, unsigned long long limit_ns,
                                         const volatile int* abort) {
  if (ld_acquire(p) >= target) return true;
  const unsigned long long t0 = globaltimer_ns();
  unsigned ns = 64;
  while (true) {
    __nanosleep(ns);
    if (ld_acquire(p) >= target) return true;
    if (*abort != 0) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      record_error(DPRC_DEVERR_READY);
      return false;
    }
    if (ns < 512) ns *= 2;
  }
}


// ---------------------------------------------------------------------------
// Thread-block clusters: ranks, distributed shared memory, remote arrivals.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// CTAs in this CTA's cluster as launched (1 for a launch without clusters).
// A kernel whose plan splits work over clusters compares it with the planned
// size before any distributed shared memory access: with another shape, a
// peer rank it would address does not exist.
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}

// All threads of every CTA in the cluster (hardware barrier; executed once,
// right after initialisation, by every thread).
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

// The two halves of cluster_sync_all, for a thread that has work to do
// before it needs its peers to have arrived (every thread of the cluster
// arrives once, then waits once, before it arrives again).
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory object in the CTA of rank `rank`.
__device__ __forceinline__ uint32_t map_to_rank(const void* local, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_u32(local)), "r"(rank));
  return out;
}

__device__ __forceinline__ void st_cluster_f4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y),
               "f"(v.z), "f"(v.w)
               : "memory");
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Asynchronous 16-byte store into another CTA's shared memory whose arrival
// is counted, as transaction bytes, on an mbarrier of that CTA (the receiver
// announces the bytes it expects with mbar_arrive_expect_tx and waits on its
// own barrier; the sender needs no fence).
__device__ __forceinline__ void st_async_f4(uint32_t cluster_addr, float4 v,
                                            uint32_t cluster_bar) {
  asm volatile(
      "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, "
      "[%5];" ::"r"(cluster_addr),
      "r"(__float_as_uint(v.x)), "r"(__float_as_uint(v.y)), "r"(__float_as_uint(v.z)),
      "r"(__float_as_uint(v.w)), "r"(cluster_bar)
      : "memory");
}

// Arrive (release at cluster scope) on an mbarrier of another CTA.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_acq_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for data that peers in the cluster published with
// mbar_arrive_remote; false (and `code` recorded) after limit_ns.
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int code,
                                                  unsigned long long limit_ns = kWaitLimitNs) {
  if (mbar_try_wait_acq_cluster(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  while (true) {
    for (int spin = 0; spin < 64; ++spin)
      if (mbar_try_wait_acq_cluster(bar, parity)) return true;
    if (globaltimer_ns() - t0 > limit_ns) {
      record_error(code);
      return false;
    }
  }
}

// ---------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor) tile loads into this CTA's shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 policy for an operand that a launch streams once: its lines are the
// first the L2 evicts, so data read again (a sketch written in L2 and read back,
// a projection matrix every CTA reads) keeps its place (PTX ISA, createpolicy).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// tma_load_3d with an L2 cache policy from l2_policy_evict_first.
__device__ __forceinline__ void tma_load_3d_hint(void* dst, const CUtensorMap* map, uint64_t* bar,
                                                 int c0, int c1, int c2, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2),
      "l"(pol)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, uint64_t* bar,
                                            int c0, int c1, int c2) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2)
      : "memory");
}

// ---------------------------------------------------------------------------
// tcgen05: tensor memory and the 5th-generation MMA.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulator; one thread issues.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive on `bar` once every MMA issued so far by this thread has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}

// Waits until every MMA this thread has issued is complete: a commit to
// `bar` (a barrier of count 1 used for nothing else, phase 0) and a bounded
// wait on it.  The MMA thread calls it last, on every path out of its loop,
// so that no MMA still writes the tensor memory the CTA releases at exit.
__device__ __forceinline__ void umma_drain(uint64_t* bar, unsigned long long limit_ns) {
  umma_commit(bar);
  mbar_wait_lim(bar, 0, DPRC_DEVERR_ACCUM, limit_ns, nullptr);
}

// 32 TMEM lanes x 32 columns of 32-bit: thread l of the warp receives lane
// (lane_base + l), columns [col, col + 32).
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

// 32 lanes x 16 columns.
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// ---------------------------------------------------------------------------
// Descriptors.
//
// Shared-memory matrix descriptor (64 bit):
//   [0,14)  start address >> 4        [16,30) leading-dimension byte offset >> 4
//   [32,46) stride-dimension byte offset >> 4     [46,48) version = 1
//   [49,52) base offset (0: atoms 1024-byte aligned)   [61,64) swizzle mode
// Swizzle modes: 0 none, 2 = 128 B, 4 = 64 B, 6 = 32 B.
//
// K-major operand with 128-byte swizzle: rows of 64 bf16 (128 B), 8-row atoms
// of 1024 B; SBO = distance between 8-row groups; LBO unused.  Successive
// K = 16 steps advance the start address by 32 B inside the swizzle row.
//
// MN-major operand with a W-byte swizzle (W = 32, 64, 128): each K row holds
// W/2 consecutive MN elements; 8 K rows form one atom of 8W bytes.  SBO =
// distance between atoms along K, LBO = distance between atoms along MN.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t make_sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                               uint32_t swz) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(swz & 7u) << 61;
  return d;
}

constexpr uint32_t kSwz128 = 2, kSwz64 = 4, kSwz32 = 6;

__host__ __device__ constexpr uint32_t swz_code_for_bytes(int bytes) {
  return bytes == 128 ? kSwz128 : (bytes == 64 ? kSwz64 : kSwz32);
}

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A/B and fp32 D:
//   [4,6) D format (1 = f32)  [7,10) A format (1 = bf16)  [10,13) B format
//   [15] A MN-major  [16] B MN-major  [17,23) N >> 3  [24,29) M >> 4
__host__ __device__ constexpr uint32_t make_idesc_bf16(int M, int N, bool a_mn, bool b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) |
         ((b_mn ? 1u : 0u) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// Named barrier among a subset of the CTA's warps.
__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t elect_one() {
  uint32_t pred = 0;
  asm volatile(
      "{\n\t.reg .b32 r;\n\t.reg .pred p;\n\t"
      "elect.sync r|p, 0xffffffff;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(pred));
  return pred;
}

// Programmatic dependent launch: wait for the previous grid's memory, and
// allow the next grid to begin its prologue.
__device__ __forceinline__ void pdl_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// bf16 hi/lo split: x ~= hi + lo with |x - hi - lo| <= 2^-17 |x|.
__device__ __forceinline__ void split_hilo(float x, __nv_bfloat16& hi, __nv_bfloat16& lo) {
  hi = __float2bfloat16_rn(x);
  lo = __float2bfloat16_rn(x - __bfloat162float(hi));
}

// A row y[0..N) as bf16 hi/lo planes [hi_0 .. hi_N-1 | lo_0 .. lo_N-1] at dst
// (16-byte aligned), 16 bytes per store.
template <int N>
__device__ __forceinline__ void store_hilo_row(__nv_bfloat16* dst, const float (&y)[N]) {
  static_assert(N % 8 == 0, "whole 16-byte chunks");
  uint32_t h[N / 2], l[N / 2];
#pragma unroll
  for (int t = 0; t < N / 2; ++t) {
    __nv_bfloat16 h0, l0, h1, l1;
    split_hilo(y[2 * t], h0, l0);
    split_hilo(y[2 * t + 1], h1, l1);
    const __nv_bfloat162 hh = __halves2bfloat162(h0, h1);
    const __nv_bfloat162 ll = __halves2bfloat162(l0, l1);
    h[t] = *reinterpret_cast<const uint32_t*>(&hh);
    l[t] = *reinterpret_cast<const uint32_t*>(&ll);
  }
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int c = 0; c < N / 8; ++c) {
    d4[c] = make_uint4(h[4 * c], h[4 * c + 1], h[4 * c + 2], h[4 * c + 3]);
    d4[N / 8 + c] = make_uint4(l[4 * c], l[4 * c + 1], l[4 * c + 2], l[4 * c + 3]);
  }
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror and Shaw, "Parallel Random Numbers: As
// Easy as 1, 2, 3", SC'11), written from that paper's definition.  Block j of
// the stream of (seed, step) is Philox applied to the counter
// (j_lo, j_hi, step_lo, step_hi) under the key (seed_lo, seed_hi).
// ---------------------------------------------------------------------------
constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

// Round keys of Philox4x32-10: the key bumped by (W0, W1) before each round.
// They depend only on the seed, so a thread computes them once.
struct RoundKeys {
  uint32_t k0[10], k1[10];
};

__device__ __forceinline__ RoundKeys round_keys(uint64_t seed) {
  RoundKeys rk;
  uint32_t a = static_cast<uint32_t>(seed), b = static_cast<uint32_t>(seed >> 32);
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    rk.k0[r] = a;
    rk.k1[r] = b;
    a += kPhiloxW0;
    b += kPhiloxW1;
  }
  return rk;
}

// Ten rounds on the counter x; each round's two 32x32 products are one wide
// multiply each (high and low words).
__device__ __forceinline__ uint4 philox4x32_10(uint4 x, const RoundKeys& rk) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    const unsigned long long p0 = static_cast<unsigned long long>(kPhiloxM0) * x.x;
    const unsigned long long p1 = static_cast<unsigned long long>(kPhiloxM1) * x.z;
    x = make_uint4(static_cast<uint32_t>(p1 >> 32) ^ x.y ^ rk.k0[r], static_cast<uint32_t>(p1),
                   static_cast<uint32_t>(p0 >> 32) ^ x.w ^ rk.k1[r], static_cast<uint32_t>(p0));
  }
  return x;
}

__device__ __forceinline__ uint4 philox_block(uint64_t j, uint64_t step, const RoundKeys& rk) {
  return philox4x32_10(make_uint4(static_cast<uint32_t>(j), static_cast<uint32_t>(j >> 32),
                                  static_cast<uint32_t>(step), static_cast<uint32_t>(step >> 32)),
                       rk);
}


// Clip factor of one squared norm v ("Method > Overall framework" of the
// notes: c = min(1, C / sqrt(n))): 1 for v = 0; 0 for a non-finite or negative
// v (an unknown norm: the sample contributes nothing), with `bad` set.
__device__ __forceinline__ float clip_factor(float v, float C, bool& bad) {
  bad = false;
  if (!isfinite(v) || v < 0.f) {
    bad = true;
    return 0.f;
  }
  if (v == 0.f) return 1.f;
  return fminf(1.f, C / sqrtf(v));
}

// Round a shared-memory pointer up to the 1024-byte alignment (of its
// shared-window address) that 128-byte swizzled tiles need.  The result is p
// plus an offset, not an integer turned back into a pointer, so the compiler
// still knows it points to shared memory and accesses through it stay
// shared-memory instructions rather than generic ones.
__device__ __forceinline__ uint8_t* align_1024(uint8_t* p) {
  return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
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

template <typename T>
__device__ __forceinline__ float to_f32(T v);
template <>
__device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

}  // namespace dprc
