// dprc_norm_hutch_noalloc: the Hutchinson estimate for callers that cannot
// allocate device memory at the call site.
//
// Some callers cannot call cudaMalloc (or any allocating routine) where they
// need the norm: code inside a framework that owns the device allocator and
// forbids direct allocations, latency-critical loops where an allocation (which
// may synchronize the device) is not acceptable, or plugins and hooks that are
// handed only their input and output pointers.  This entry point takes no
// workspace: its scratch is a fixed-size array in the library's own device
// memory, reserved on every GPU that loads the library until the process exits.
//
// There is no counterpart on the method's pages; the method does not discuss
// memory allocation.

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "dprc.h"
#include "internal.h"

namespace {

// The shared scratch.  In host code this name is only a host-side stand-in:
// the device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DPRC_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
dprc_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DPRC_ERR_DEVICE;
  if (dev < 0 || dev >= kMaxDevices) return DPRC_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      (void)cudaGetLastError();  // leave no sticky error behind for the caller
      return DPRC_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return DPRC_OK;
}

}  // namespace

extern "C" dprc_status dprc_norm_hutch_noalloc(const void* A, const void* G, const void* P,
                                               dprc_dtype dtype, int64_t B, int64_t T,
                                               int64_t d, int64_t p, int64_t k, float* n,
                                               int accumulate, void* stream) {
  DPRC_NVTX_RANGE();
  // every check that needs no device first: an argument error returns before
  // the scratch is looked up or its counters are cleared
  dprc_status st = dprc::check_hutch_args(A, G, P, dtype, B, T, d, p, k, n);
  if (st != DPRC_OK) return st;
  const size_t need = dprc_workspace_bytes(DPRC_OP_HUTCH, dtype, B, T, d, p, k);
  if (need == 0) return DPRC_ERR_SHAPE;
  if (need > static_cast<size_t>(DPRC_NOALLOC_SCRATCH_BYTES)) return DPRC_ERR_TOO_LARGE;
  if (!dprc::current_device_supported()) return DPRC_ERR_DEVICE;
  void* ws = nullptr;
  st = scratch_address(&ws);
  if (st != DPRC_OK) return st;
  // the counters at the front of the scratch must start at zero
  if (cudaMemsetAsync(ws, 0, dprc::ctrl_bytes(B), static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return DPRC_ERR_CUDA;
  return dprc_norm_hutch(A, G, P, dtype, B, T, d, p, k, n, accumulate, ws,
                         static_cast<size_t>(DPRC_NOALLOC_SCRATCH_BYTES), stream);
}
